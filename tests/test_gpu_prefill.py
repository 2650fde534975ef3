"""Multi-query paged attention (chunked prefill, decode tokens in the same
batch) on the GPU against the fp64 oracle: element-wise
|gpu - oracle| <= 4e-3 + 1e-2 |oracle| over head_dim, dtype, group size and
block size; chunks of 1 token (decode), fewer than a tile, exactly a tile and
many tiles; empty and unaligned cached prefixes; NaN in every slot the step
does not read.  Plus: bit-identical repeats through one workspace, a batch of
decode tokens against the decode oracle, invalid sequences reported with zero
rows, and sampled parity on the Llama-3-8B chunked-prefill step."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState, OracleState, assert_close, check_parity, gpu_out_f64, gpu_step
from paged_kv_cache_72_gb300 import _lib

pytestmark = pytest.mark.gpu

PREFIX = [0, 0, 5, 63, 64, 100, 700, 1500]
CHUNK = [1, 37, 1, 64, 200, 5, 129, 300]


def _parity(wl):
    st = GpuState(wl)
    out, _ = gpu_step(st)
    ref = OracleState(wl)
    ref.step()
    expected, spread = ref.decode(spread=True)
    check_parity(out, wl, expected, spread, wl.name)
    assert pa.pa_get_error(st.err) == 0
    return st, out


CASES = [
    # dtype, Hq, Hkv, D, B
    (W.BF16, 32, 8, 128, 16),   # the Llama-3-8B shape: 32 tokens x 4 heads per item
    (W.F16, 8, 8, 128, 16),     # G = 1: 128 tokens per item
    (W.BF16, 16, 2, 64, 16),    # G = 8
    (W.F16, 14, 2, 64, 8),      # G = 7: 18 tokens, two padding rows per item
    (W.BF16, 32, 2, 128, 32),   # G = 16
    (W.F16, 6, 3, 128, 4),
    (W.BF16, 12, 4, 64, 256),
    (W.BF16, 16, 4, 128, 8),    # V boxes of 8 rows x 2 planes: 8-key groups one block apart
    (W.F16, 8, 2, 128, 64),     # one 64-row block per stage
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B", CASES)
def test_prefill_parity_sweep(cuda_device, dtype, Hq, Hkv, D, B):
    wl = W.random_prefill(130 + Hq + B, dtype, Hq, Hkv, D, B, PREFIX, CHUNK, garbage="nan")
    _parity(wl)


def test_prefill_kernel_choice(cuda_device):
    # Every shape with blocks of 8 or more tokens runs the tensor-core kernel,
    # at any batch size; blocks of 4 tokens (head_dim 128) take the
    # warp-level kernel.
    # A tensor-core plan that stops fitting the device (registers, shared
    # memory) would otherwise fall back to the slower kernel with every
    # parity test still passing.
    for dtype in (W.F16, W.BF16):
        for D in (64, 128):
            for B in (8, 16, 64, 256):
                for (Hq, Hkv) in ((32, 8), (14, 2), (8, 8)):
                    for n in (1, 16, 4096):
                        assert pa.pa_prefill_kernel(Hq, Hkv, D, B, dtype, n) == \
                            pa.PA_PREFILL_TENSOR_CORE, (dtype, D, B, Hq, Hkv, n)
    assert pa.pa_prefill_kernel(8, 2, 128, 4, W.F16, 6) == pa.PA_PREFILL_WARP_MMA
    assert pa.pa_prefill_kernel(8, 8, 128, 4, W.BF16, 4096) == pa.PA_PREFILL_WARP_MMA
    for shape in ((8, 2, 96, 16), (8, 2, 128, 2), (8, 2, 64, 4)):   # refused by pa_prefill too
        with pytest.raises(pa.PAError):
            pa.pa_prefill_kernel(*shape, W.F16, 6)


def test_prefill_repeats_bitwise_through_one_workspace(cuda_device):
    wl = W.random_prefill(140, W.BF16, 32, 8, 128, 16, PREFIX, CHUNK)
    st, out = _parity(wl)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    a = pa.pa_prefill(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, st.query_start,
                      wl.scale, workspace=ws)
    b = pa.pa_prefill(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, st.query_start,
                      wl.scale, workspace=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), out.view(torch.int16))
    assert not ws.any()   # the work counters are back at zero
    # and no call sits out a wait bound (about 2 s): ten calls take far less
    import time
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(10):
        pa.pa_prefill(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                      st.query_start, wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0


def test_prefill_of_single_tokens_is_the_decode(cuda_device):
    lens = [1, 16, 17, 300, 2049]
    wl = W.random_prefill(141, W.F16, 8, 2, 128, 16, [t - 1 for t in lens], [1] * len(lens))
    st = GpuState(wl)
    out, _ = gpu_step(st)
    ref = OracleState(wl)
    ref.step()
    dec = oracle.paged_decode(wl.q, ref.k_cache, ref.v_cache, wl.dtype, wl.block_tables,
                              wl.seq_lens, wl.scale)
    assert_close(gpu_out_f64(out), dec, "single tokens vs decode")


def test_prefill_reports_invalid_sequences(cuda_device):
    wl = W.random_prefill(142, W.BF16, 8, 2, 64, 16, [10, 40], [5, 20])
    st = GpuState(wl)
    gpu_step(st, decode=False)
    bad = torch.tensor([3, 60], dtype=torch.int32, device="cuda")   # 5 new tokens but T = 3
    out = pa.pa_prefill(st.q, st.k_cache, st.v_cache, st.block_tables, bad, st.query_start,
                        wl.scale, err=st.err)
    assert pa.pa_get_error(st.err) == pa.PA_DEVERR_SEQ_LEN
    assert not out[:5].any()


def test_llama3_chunked_prefill_sampled(cuda_device):
    wl = W.llama3_8b_chunked_prefill()
    st = GpuState(wl)
    out, _ = gpu_step(st)
    assert pa.pa_get_error(st.err) == 0
    ref = OracleState(wl)
    ref.step()
    # the oracle on two sequences (their rows), the shortest and the longest prefix
    order = np.argsort(wl.seq_lens)
    for i in (int(order[0]), int(order[-1])):
        q0, q1 = wl.query_start[i], wl.query_start[i + 1]
        sub, sp = oracle.paged_prefill(wl.q[q0:q1], ref.k_cache, ref.v_cache, wl.dtype,
                                       wl.block_tables[i:i + 1], wl.seq_lens[i:i + 1],
                                       np.array([0, q1 - q0], np.int32), wl.scale, spread=True)
        check_parity(out[q0:q1], wl, sub, sp, "llama3 chunked prefill seq %d" % i)


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_wide_score_range(cuda_device, D):
    """q, k ~ N(0, 4^2): scores spread over tens of binary orders, so a row's
    running maximum moves past the kernel's reference many times and its rows
    of O are rescaled in tensor memory.

    On such peaked rows the 16-bit P costs more than the plain decode
    tolerance allows.  With P_i rounded to p_i (1 + d_i), |d_i| <= 2^-8
    (bfloat16), the output moves by sum_i p_i d_i (v_i - out) / sum_i p_i, at
    most 2^-8 * 2 max|v|, and its own rounding adds at most 2^-8 |out|: the
    coarse bound below.  The rounding bound (the same terms per element, with
    the oracle's weighted deviation in place of 2 max|v|) must hold too."""
    wl = W.random_prefill(150 + D, W.BF16, 16, 4, D, 16, [0, 500, 2000, 63], [300, 129, 64, 70],
                          garbage="nan", q_sigma=4.0, kv_sigma=4.0)
    st = GpuState(wl)
    out, _ = gpu_step(st)
    ref = OracleState(wl)
    ref.step()
    expected = ref.decode()
    assert pa.pa_get_error(st.err) == 0
    got = gpu_out_f64(out)
    assert np.all(np.isfinite(got))
    vmax = max(float(np.abs(oracle.gather_head(ref.v_cache, wl.dtype, wl.block_tables[i],
                                                   int(wl.seq_lens[i]), h)).max())
               for i in range(len(wl.seq_lens)) for h in range(wl.num_kv_heads))
    bound = 4e-3 + 1e-2 * np.abs(expected) + 3 * 2.0 ** -8 * vmax
    assert np.all(np.abs(got - expected) <= bound), float(np.abs(got - expected).max())
    _, spread = ref.decode(spread=True)
    check_parity(out, wl, expected, spread, "wide score range D=%d" % D, allclose=False)


def test_prefill_sequences_ending_on_stage_edges(cuda_device):
    # lengths at, one past and one short of multiples of the 64-key stage, so
    # the V rows past the end are cleared in some stages and in none of others
    prefix = [64 - 5, 128 - 1, 191, 256 - 64, 0, 1]
    chunk = [5, 1, 2, 64, 64, 63]
    wl = W.random_prefill(160, W.F16, 8, 2, 128, 16, prefix, chunk, garbage="nan")
    _parity(wl)


@pytest.mark.parametrize("n", [192, 193])
def test_prefill_item_order_either_side_of_the_rank_limit(cuda_device, n):
    # up to 192 sequences the tensor-core kernel takes its items longest
    # sequence first (ranked in shared memory, ties by index), past that in
    # batch order; both must cover every item once
    rng = np.random.default_rng(n)
    prefix = rng.integers(0, 150, size=n)
    chunk = rng.integers(1, 40, size=n)
    prefix[::5] = 64 - chunk[::5]   # ties: every fifth sequence 64 tokens long
    wl = W.random_prefill(170 + n, W.BF16, 16, 4, 128, 16, prefix, chunk, garbage="nan")
    assert pa.pa_prefill_kernel(16, 4, 128, 16, W.BF16, n) == pa.PA_PREFILL_TENSOR_CORE
    _parity(wl)


def test_prefill_at_the_sequence_limit(cuda_device):
    # every sequence's item offset sits in shared memory, up to 4,096
    # sequences: a batch of 4,096, mostly single decode tokens with a chunk in
    # every 97th, and one sequence more is refused
    rng = np.random.default_rng(4096)
    n = 4096
    prefix = rng.integers(0, 60, size=n)
    chunk = np.ones(n, dtype=np.int64)
    chunk[::97] = rng.integers(2, 40, size=chunk[::97].size)
    wl = W.random_prefill(4096, W.BF16, 8, 2, 64, 16, prefix, chunk, garbage="nan")
    _parity(wl)
    st = GpuState(wl)
    extra_lens = torch.cat([st.seq_lens, st.seq_lens[:1]])
    extra_qs = torch.cat([st.query_start, st.query_start[-1:] + 1])
    q = torch.zeros((int(wl.query_start[-1]) + 1,) + tuple(st.q.shape[1:]), dtype=st.q.dtype,
                    device="cuda")
    bt = torch.cat([st.block_tables, st.block_tables[:1]])
    with pytest.raises(pa.PAError) as e:
        pa.pa_prefill(q, st.k_cache, st.v_cache, bt, extra_lens, extra_qs, wl.scale, err=st.err)
    assert e.value.status == _lib.PA_ERR_UNSUPPORTED
