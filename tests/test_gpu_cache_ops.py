"""Slot mapping, cache write and copy-on-write block copy on the GPU, compared
bit for bit with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState, OracleState, bits_of, gpu_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [W.tiny, W.shared_prefix])
def test_step_writes_are_bit_exact(cuda_device, make):
    wl = make()
    st = GpuState(wl)
    _, slots = gpu_step(st, decode=False)
    ref = OracleState(wl)
    ref.step()
    assert np.array_equal(slots.cpu().numpy(), ref.slots)
    assert np.array_equal(bits_of(st.k_cache), ref.k_cache)
    assert np.array_equal(bits_of(st.v_cache), ref.v_cache)
    assert pa.pa_get_error(st.err) == 0


def test_shared_prefix_sharers_read_identical_prefix(cuda_device):
    # sequences sharing blocks see the same K/V ("vLLM": requests point at the
    # same blocks); after the copy-on-write the 8 prefix tokens of the copied
    # block are identical too
    wl = W.shared_prefix()
    st = GpuState(wl)
    gpu_step(st, decode=False)
    k = bits_of(st.k_cache)
    first = [oracle.gather_bits(k, wl.block_tables[i], 1800) for i in range(wl.num_seqs)]
    for g in first[1:]:
        assert np.array_equal(g, first[0])


def test_slot_mapping_random_positions(cuda_device):
    rng = np.random.default_rng(40)
    nb, B, N, stride = 500, 16, 37, 20
    bt = rng.integers(0, nb, size=(N, stride)).astype(np.int32)
    seq = rng.integers(0, N, size=3000).astype(np.int32)
    pos = rng.integers(0, stride * B, size=3000).astype(np.int32)
    got = pa.pa_slot_mapping(torch.from_numpy(bt).cuda(), torch.from_numpy(seq).cuda(),
                             torch.from_numpy(pos).cuda(), B, nb)
    assert np.array_equal(got.cpu().numpy(), oracle.slot_mapping(bt, seq, pos, B))


def test_slot_mapping_flags_bad_positions(cuda_device):
    bt = torch.tensor([[3, 1], [0, 2]], dtype=torch.int32, device="cuda")
    seq = torch.tensor([0, 1, 2, 0, 1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([5, 7, 0, 8, -1], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pa.pa_slot_mapping(bt, seq, pos, 4, 4, err=err)
    assert got.cpu().tolist() == [5, 11, -1, -1, -1]
    assert pa.pa_get_error(err) == pa.PA_DEVERR_POSITION
    bt_bad = torch.tensor([[3, 9]], dtype=torch.int32, device="cuda")
    got = pa.pa_slot_mapping(bt_bad, seq[:1] * 0, torch.tensor([6], dtype=torch.int32,
                                                                  device="cuda"), 4, 4, err=err)
    assert got.cpu().tolist() == [-1]
    assert pa.pa_get_error(err) == pa.PA_DEVERR_BLOCK_ID


def test_cache_write_padding_and_out_of_range_slots(cuda_device):
    rng = np.random.default_rng(41)
    nb, B, H, D = 6, 4, 2, 64
    kc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    k = rng.integers(0, 65535, size=(4, H, D), dtype=np.uint16)
    v = rng.integers(0, 65535, size=(4, H, D), dtype=np.uint16)
    slots = np.array([3, -1, nb * B, 23], np.int64)
    dk = torch.from_numpy(kc.view(np.int16)).cuda().view(torch.float16)
    dv = torch.from_numpy(vc.view(np.int16)).cuda().view(torch.float16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_cache_write(torch.from_numpy(k.view(np.int16)).cuda().view(torch.float16),
                      torch.from_numpy(v.view(np.int16)).cuda().view(torch.float16),
                      torch.from_numpy(slots).cuda(), dk, dv, err=err)
    assert pa.pa_get_error(err) == pa.PA_DEVERR_SLOT
    ok = slots.copy()
    ok[2] = -1
    oracle.cache_write(kc, vc, k, v, ok)
    assert np.array_equal(bits_of(dk), kc) and np.array_equal(bits_of(dv), vc)


def test_copy_blocks_rejects_conflicting_pairs(cuda_device):
    rng = np.random.default_rng(42)
    nb, B, H, D = 10, 16, 2, 64
    kc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    dk = torch.from_numpy(kc.view(np.int16)).cuda().view(torch.bfloat16)
    dv = torch.from_numpy(vc.view(np.int16)).cuda().view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # (4 -> 5) writes a block that (5 -> 6) reads, so it is dropped; (1 -> 12)
    # is out of range; (3 -> 9) and (0 -> 9) repeat a dst, both dropped
    pairs = np.array([[0, 7], [4, 5], [5, 6], [1, 12], [2, 8], [3, 9], [0, 9]], np.int32)
    pa.pa_copy_blocks(torch.from_numpy(pairs).cuda(), dk, dv, err=err)
    assert pa.pa_get_error(err) == pa.PA_DEVERR_COPY_PAIR
    oracle.copy_blocks(kc, vc, np.array([[0, 7], [5, 6], [2, 8]], np.int32))
    assert np.array_equal(bits_of(dk), kc) and np.array_equal(bits_of(dv), vc)


def test_empty_calls_are_no_ops(cuda_device):
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.float16, device="cuda")
    out = pa.pa_slot_mapping(torch.zeros((1, 1), dtype=torch.int32, device="cuda"), z, z, 16, 4)
    assert out.numel() == 0
    pa.pa_copy_blocks(torch.zeros((0, 2), dtype=torch.int32, device="cuda"), kc, kc.clone())
    pa.pa_cache_write(torch.zeros((0, 2, 64), dtype=torch.float16, device="cuda"),
                      torch.zeros((0, 2, 64), dtype=torch.float16, device="cuda"),
                      torch.zeros(0, dtype=torch.int64, device="cuda"), kc, kc.clone())
    torch.cuda.synchronize()


@pytest.mark.parametrize("make", [W.tiny, W.shared_prefix,
                                  lambda: W.random_workload(44, W.BF16, 32, 8, 128, 16,
                                                            [1, 16, 17, 300, 777])])
def test_slot_mapped_cache_write_is_bit_exact(cuda_device, make):
    # the one-launch slot mapping + cache write stores the same bytes and
    # returns the same slots as the oracle's scatter ("vLLM Framework and
    # Inference Engine Design", "How is vLLM's KV cache paged?", "Writing")
    wl = make()
    st = GpuState(wl)
    ref = OracleState(wl)
    ref.step()
    if st.pairs.numel():
        pa.pa_copy_blocks(st.pairs, st.k_cache, st.v_cache, err=st.err)
    slots = torch.full((wl.new_seq.size,), 7, dtype=torch.int64, device="cuda")
    pa.pa_cache_write_mapped(st.k_new, st.v_new, st.block_tables, st.new_seq, st.new_pos,
                             st.k_cache, st.v_cache, slot_mapping=slots, err=st.err)
    assert np.array_equal(slots.cpu().numpy(), ref.slots)
    assert np.array_equal(bits_of(st.k_cache), ref.k_cache)
    assert np.array_equal(bits_of(st.v_cache), ref.v_cache)
    assert pa.pa_get_error(st.err) == 0


def test_slot_mapped_cache_write_flags_bad_tokens(cuda_device):
    # bad sequence index, position or table entry: slot -1, nothing written,
    # the same error bits as the slot mapping
    H, D, B, nb = 2, 64, 4, 4
    bt = torch.tensor([[3, 1], [0, 9]], dtype=torch.int32, device="cuda")
    seq = torch.tensor([0, 1, 2, 0, 1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([5, 1, 0, -1, 6], dtype=torch.int32, device="cuda")
    k = torch.randn(5, H, D, device="cuda").to(torch.float16)
    v = torch.randn(5, H, D, device="cuda").to(torch.float16)
    kc = torch.zeros(nb, B, H, D, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.zeros(5, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_cache_write_mapped(k, v, bt, seq, pos, kc, vc, slot_mapping=slots, err=err)
    assert slots.cpu().tolist() == [5, 1, -1, -1, -1]
    assert pa.pa_get_error(err) == pa.PA_DEVERR_POSITION | pa.PA_DEVERR_BLOCK_ID
    kf, vf = kc.view(nb * B, H, D), vc.view(nb * B, H, D)
    assert torch.equal(kf[5], k[0]) and torch.equal(vf[5], v[0])
    assert torch.equal(kf[1], k[1]) and torch.equal(vf[1], v[1])
    written = torch.zeros(nb * B, dtype=torch.bool)
    written[[1, 5]] = True
    assert not kf[~written.cuda()].any() and not vf[~written.cuda()].any()
    # without a slot output the pools end the same
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(vc)
    pa.pa_cache_write_mapped(k, v, bt, seq, pos, kc2, vc2)
    assert torch.equal(kc2, kc) and torch.equal(vc2, vc)


def _valid_pairs(pairs, nb):
    """The pairs the block copy must apply: in range, dst unique among the
    dsts and no pair's src (the rules stated for pa_copy_blocks)."""
    src, dst = pairs[:, 0], pairs[:, 1]
    ok = (src >= 0) & (src < nb) & (dst >= 0) & (dst < nb)
    uniq, counts = np.unique(dst, return_counts=True)
    dup = set(uniq[counts > 1].tolist())
    srcs = set(src.tolist())
    ok &= np.array([d not in dup and d not in srcs for d in dst.tolist()])
    return pairs[ok]


def test_copy_blocks_4096_pairs_with_conflicts_far_apart(cuda_device):
    # a fork of many samples: 4,096 pairs, handled by many thread blocks; the
    # conflicting pairs sit far apart in the list, in other blocks' ranges
    rng = np.random.default_rng(45)
    n, nb, B, H, D = 4096, 9000, 16, 2, 64
    kc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    perm = rng.permutation(nb).astype(np.int32)
    pairs = np.stack([perm[:n], perm[n:2 * n]], 1).astype(np.int32)
    pairs[10, 1] = pairs[4000, 1]      # one dst twice: both dropped
    pairs[20, 1] = pairs[3000, 0]      # a dst that another pair reads: dropped
    pairs[30, 0] = nb + 5              # out of range: dropped
    pairs[2000, 1] = pairs[2000, 0]    # a block onto itself (its dst is a src): dropped
    valid = _valid_pairs(pairs, nb)
    assert valid.shape[0] == n - 5
    dk = torch.from_numpy(kc.view(np.int16)).cuda().view(torch.float16)
    dv = torch.from_numpy(vc.view(np.int16)).cuda().view(torch.float16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(torch.from_numpy(pairs).cuda(), dk, dv, err=err)
    assert pa.pa_get_error(err) == pa.PA_DEVERR_COPY_PAIR
    oracle.copy_blocks(kc, vc, valid)
    assert np.array_equal(bits_of(dk), kc) and np.array_equal(bits_of(dv), vc)


def test_copy_blocks_time_grows_linearly_with_pairs(cuda_device):
    # each thread block validates its own pairs against one pass over the list,
    # so the call's time grows with the number of pairs, not with its square
    nb, B, H, D = 17000, 16, 1, 64
    kc = torch.zeros((nb, B, H, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    perm = np.random.default_rng(46).permutation(nb).astype(np.int32)
    times = {}
    for n in (512, 2048, 8192):
        pairs = torch.from_numpy(np.stack([perm[:n], perm[n:2 * n]], 1).copy()).cuda()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ms = []
        for rep in range(9):
            ev[0].record()
            pa.pa_copy_blocks(pairs, kc, vc, err=err)
            ev[1].record()
            torch.cuda.synchronize()
            if rep >= 2:
                ms.append(ev[0].elapsed_time(ev[1]))
        times[n] = sorted(ms)[len(ms) // 2]
    assert pa.pa_get_error(err) == 0
    # 16 times the pairs: a quadratic check would take over 100 times as long
    assert times[8192] < 16 * times[512] + 0.05, times
