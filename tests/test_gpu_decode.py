"""Paged decode attention on the GPU against the fp64 oracle: element-wise
|gpu - oracle| <= 4e-3 + 1e-2 |oracle|, over head_dim, dtype, group size,
block size, ragged lengths (empty, one token, block and chunk edges), grid
sizes that split contexts across thread blocks, both kernels, garbage (NaN) in
unread slots; plus the properties the pages fix: the result does not depend
on where blocks sit, and equals unpaged attention."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import (GpuState, OracleState, assert_close, bits_of, check_parity, gpu_out_f64,
                     gpu_step, to_dev)

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 200, 777]


def _parity(wl, flags=pa.PA_DECODE_AUTO, num_ctas=0):
    st = GpuState(wl)
    out, _ = gpu_step(st, flags=flags, num_ctas=num_ctas)
    ref = OracleState(wl)
    ref.step()
    expected, spread = ref.decode(spread=True)
    rep = check_parity(out, wl, expected, spread,
                       "%s flags=%d ctas=%d" % (wl.name, flags, num_ctas), flags=flags)
    assert pa.pa_get_error(st.err) == 0
    return out, rep["max_abs"]


def test_tiny_config(cuda_device):
    wl = W.tiny()
    _parity(wl)
    _parity(wl, flags=pa.PA_DECODE_MMA)


CASES = [
    # dtype, Hq, Hkv, D, B
    (W.F16, 4, 4, 128, 16),
    (W.BF16, 4, 4, 64, 16),
    (W.BF16, 8, 2, 128, 16),
    (W.F16, 8, 2, 64, 16),
    (W.BF16, 14, 2, 64, 16),
    (W.F16, 14, 2, 128, 8),
    (W.BF16, 16, 2, 128, 16),
    (W.F16, 16, 1, 64, 32),
    (W.BF16, 32, 2, 128, 16),
    (W.F16, 6, 3, 128, 4),
    (W.BF16, 4, 2, 128, 2),
    (W.BF16, 8, 8, 128, 128),
    (W.F16, 12, 4, 64, 256),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B", CASES)
def test_parity_sweep(cuda_device, dtype, Hq, Hkv, D, B):
    wl = W.random_workload(1000 + Hq * 7 + D + B, dtype, Hq, Hkv, D, B, EDGE_LENS,
                           kv_sigma=0.7, garbage="nan")
    _parity(wl)
    if Hq == Hkv:
        _parity(wl, flags=pa.PA_DECODE_MMA)


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 50, 1000])
def test_split_contexts_across_blocks(cuda_device, num_ctas):
    # few blocks: long ranges spanning many sequences; many blocks (more than
    # the GPU holds at once): contexts split into one-chunk pieces, each merged
    # by whichever block's piece arrives last
    lens = [3000, 1, 64, 65, 900, 2048, 5, 4096]
    wl = W.random_workload(77, W.BF16, 16, 4, 128, 16, lens, kv_sigma=0.5)
    _parity(wl, num_ctas=num_ctas)
    wl1 = W.random_workload(78, W.F16, 4, 4, 128, 16, lens)
    _parity(wl1, num_ctas=num_ctas)


def test_one_workspace_across_calls_that_split_differently(cuda_device):
    # the split-merge counters live in the workspace and every call must leave
    # them at zero: one workspace serves calls whose contexts split at other
    # places (grid sizes from 1 to more than the GPU holds, other lengths)
    lens = [3000, 1, 64, 65, 900, 2048, 5, 4096]
    wl = W.random_workload(21, W.BF16, 16, 4, 128, 16, lens, kv_sigma=0.5)
    st = GpuState(wl)
    gpu_step(st, decode=False)
    ref = OracleState(wl)
    ref.step()
    full = ref.decode()
    short = np.array([1500, 1, 33, 65, 17, 2048, 5, 999], np.int32)
    exp_short = oracle.paged_decode(wl.q, ref.k_cache, ref.v_cache, wl.dtype, wl.block_tables,
                                    short, wl.scale)
    sl_short = torch.from_numpy(short).cuda()
    sizes = [0, 7, 1000, 3, 152, 50, 1, 0]
    nbytes = max(pa.pa_decode_workspace_size(16, 4, 128, 16, torch.bfloat16, num_ctas=n)
                 for n in sizes)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for k, n in enumerate(sizes):
        sl, expected = (st.seq_lens, full) if k % 2 == 0 else (sl_short, exp_short)
        out = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, sl, wl.scale,
                           workspace=ws, num_ctas=n, err=st.err)
        assert_close(gpu_out_f64(out), expected, "call %d, ctas=%d" % (k, n))
    assert pa.pa_get_error(st.err) == 0


def test_placement_does_not_change_bits(cuda_device):
    # the same logical cache in two physical arrangements gives identical bits
    lens = [5, 700, 64, 1300]
    B, H, D = 16, 2, 128
    base = W.random_workload(5, W.BF16, 8, H, D, B, lens, num_blocks=300)
    outs = []
    for seed in (0, 1):
        perm = np.random.default_rng(seed).permutation(base.num_blocks).astype(np.int32)
        kc = np.zeros_like(base.k_cache)
        vc = np.zeros_like(base.v_cache)
        used = base.block_tables >= 0
        kc[perm[base.block_tables[used]]] = base.k_cache[base.block_tables[used]]
        vc[perm[base.block_tables[used]]] = base.v_cache[base.block_tables[used]]
        bt = np.where(used, perm[np.maximum(base.block_tables, 0)], -1).astype(np.int32)
        q = to_dev(base.q, base.dtype)
        out = pa.pa_decode(q, to_dev(kc, base.dtype), to_dev(vc, base.dtype),
                           torch.from_numpy(bt).cuda(), torch.from_numpy(base.seq_lens).cuda(),
                           base.scale)
        outs.append(bits_of(out))
    assert np.array_equal(outs[0], outs[1])


def test_identity_placement_equals_contiguous_attention(cuda_device):
    T, Hq, H, D, B = 1000, 8, 2, 128, 16
    nb = -(-T // B)
    wl = W.random_workload(9, W.F16, Hq, H, D, B, [T], num_blocks=nb)
    bt = np.arange(nb, dtype=np.int32)[None, :]
    out = pa.pa_decode(to_dev(wl.q, wl.dtype), to_dev(wl.k_cache, wl.dtype),
                       to_dev(wl.v_cache, wl.dtype), torch.from_numpy(bt).cuda(),
                       torch.tensor([T], dtype=torch.int32, device="cuda"), wl.scale)
    K = oracle.decode(wl.k_cache, W.F16).reshape(nb * B, H, D)[:T]
    V = oracle.decode(wl.v_cache, W.F16).reshape(nb * B, H, D)[:T]
    ref = oracle.contiguous_decode(oracle.decode(wl.q[0], W.F16), K, V, wl.scale)
    assert_close(gpu_out_f64(out)[0], ref, "contiguous")


def test_repeat_runs_are_bitwise_identical(cuda_device):
    wl = W.random_workload(11, W.BF16, 32, 8, 128, 16, [100, 4000, 37, 600])
    st = GpuState(wl)
    a = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale)
    b = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_zero_and_invalid_lengths(cuda_device):
    lens = [0, 40, 0, 17]
    wl = W.random_workload(12, W.F16, 8, 2, 64, 16, [1, 40, 1, 17])
    st = GpuState(wl)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, sl, wl.scale, err=st.err)
    assert pa.pa_get_error(st.err) == 0
    o = gpu_out_f64(out)
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    ref = oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                              np.array(lens, np.int32), wl.scale)
    assert_close(o, ref, "zero lengths")
    # a length beyond the table row and a negative one are reported, and their
    # rows are zero; the others are unaffected
    bad = torch.tensor([-3, 40, 10 ** 6, 17], dtype=torch.int32, device="cuda")
    out = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, bad, wl.scale, err=st.err)
    assert pa.pa_get_error(st.err) == pa.PA_DEVERR_SEQ_LEN
    o = gpu_out_f64(out)
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert_close(o[[1, 3]], ref[[1, 3]], "valid rows next to invalid ones")


def test_bad_block_id_is_reported_not_faulted(cuda_device):
    wl = W.random_workload(13, W.BF16, 8, 2, 128, 16, [50, 50])
    st = GpuState(wl)
    bt = st.block_tables.clone()
    bt[1, 1] = wl.num_blocks + 5
    bt[0, 0] = -7
    pa.pa_decode(st.q, st.k_cache, st.v_cache, bt, st.seq_lens, wl.scale, err=st.err)
    assert pa.pa_get_error(st.err) == pa.PA_DEVERR_BLOCK_ID


def test_alternating_shapes_of_one_kernel(cuda_device):
    # group sizes 4 and 2 run the same kernel with different shared-memory
    # layouts; calling them in turn must keep working
    a = W.random_workload(15, W.BF16, 8, 2, 128, 16, [300, 5])
    b = W.random_workload(16, W.BF16, 4, 2, 128, 16, [70, 900, 1])
    for wl in (a, b, a, b):
        _parity(wl)


def test_empty_batch(cuda_device):
    q = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 16, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = pa.pa_decode(q, kc, kc.clone(), torch.zeros((0, 1), dtype=torch.int32, device="cuda"),
                       torch.zeros(0, dtype=torch.int32, device="cuda"), 0.1)
    assert out.shape == (0, 8, 128)


def test_workspace_too_small(cuda_device):
    wl = W.random_workload(14, W.BF16, 8, 2, 128, 16, [50])
    st = GpuState(wl)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale,
                     workspace=ws)
    assert e.value.status == 3


@pytest.mark.parametrize("flags", [pa.PA_DECODE_SIMT, pa.PA_DECODE_MMA])
@pytest.mark.parametrize("B,D,dtype", [(4, 64, W.F16), (16, 128, W.BF16), (32, 64, W.BF16),
                                       (2, 128, W.F16), (128, 128, W.F16)])
def test_gather_is_bit_exact(cuda_device, flags, B, D, dtype):
    lens = [1, B - 1 if B > 1 else 1, B, B + 1, 63, 64, 65, 300]
    wl = W.random_workload(200 + B + D, dtype, 2, 2, D, B, lens, garbage="nan")
    st = GpuState(wl)
    offs = np.concatenate([[0], np.cumsum(wl.seq_lens)[:-1]]).astype(np.int64)
    k_out, v_out = pa.pa_gather_kv(st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                                   torch.from_numpy(offs).cuda(), int(wl.seq_lens.sum()),
                                   flags=flags, err=st.err)
    assert pa.pa_get_error(st.err) == 0
    kg, vg = bits_of(k_out), bits_of(v_out)
    for i, T in enumerate(wl.seq_lens):
        o = offs[i]
        assert np.array_equal(kg[o:o + T], oracle.gather_bits(wl.k_cache, wl.block_tables[i], T))
        assert np.array_equal(vg[o:o + T], oracle.gather_bits(wl.v_cache, wl.block_tables[i], T))


@pytest.mark.parametrize("kind", ["bf16", "fp8", "window"])
def test_more_sequences_than_the_length_cache(cuda_device, kind):
    # the decode keeps the first 1,024 lengths in shared memory and reads the
    # others from global memory: 2,500 short sequences cross that line, with
    # the lengths and tables read before the grid-dependency wait
    rng = np.random.default_rng(2500)
    lens = rng.integers(1, 80, size=2500)
    lens[[0, 1023, 1024, 1025, 2499]] = [1, 17, 33, 1, 79]
    kw = {"fp8": {"fp8_scales": (2.0 ** -6, 2.0 ** -6)}, "window": {"window": 20}}.get(kind, {})
    wl = W.random_workload(2500, W.BF16, 8, 2, 64, 16, lens, kv_sigma=0.7, garbage="nan", **kw)
    flags = pa.PA_DECODE_TABLES_READY
    st = GpuState(wl)
    out, _ = gpu_step(st, flags=flags)
    assert pa.pa_get_error(st.err) == 0
    ref = OracleState(wl)
    ref.step()
    expected, spread = ref.decode(spread=True)
    check_parity(out, wl, expected, spread, "%s, 2,500 sequences" % kind, flags=flags)
