"""Host-side checks of the seeded workload generators and block bookkeeping,
against the facts the pages fix for paging (ceil(T/B) blocks, fewer than B
wasted slots, blocks anywhere in the pool, reference counts, copy-on-write)."""
import numpy as np
import pytest

import oracle
import workloads as W
from workloads.blocks import BlockPool, Sequence


def _check_tables(wl):
    B = wl.block_size
    seen = set()
    for i, T in enumerate(wl.seq_lens):
        n = oracle.blocks_for(int(T), B)
        row = wl.block_tables[i]
        assert np.all(row[:n] >= 0) and np.all(row[:n] < wl.num_blocks)
        assert np.all(row[n:] == -1)
        assert n * B - int(T) < B
        for p in row[:n]:
            seen.add(int(p))
    return seen


def test_tiny_shape_and_tables():
    wl = W.tiny()
    assert wl.seq_lens.tolist() == [7, 8, 9, 33]
    assert (wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size) == (8, 8, 64, 4)
    used = _check_tables(wl)
    # 2 + 2 + 3 + 9 distinct blocks of the 32-block pool
    assert len(used) == 16
    assert wl.new_pos.tolist() == [6, 7, 8, 32]


def test_generators_are_deterministic():
    a, b = W.tiny(seed=9), W.tiny(seed=9)
    for f in ("q", "k_cache", "v_cache", "block_tables", "k_new", "v_new"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    c = W.tiny(seed=10)
    assert not np.array_equal(a.q, c.q)


def test_llama3_lengths_distribution():
    lens = W.llama3_8b_lengths()
    assert lens.shape == (256,)
    assert lens.min() >= 16 and lens.max() <= 4096
    assert 340 <= lens.mean() <= 460


def test_shared_prefix_copy_on_write_plan():
    wl = W.shared_prefix()
    B = wl.block_size
    prefix_blocks = oracle.blocks_for(1800, B)
    assert prefix_blocks == 113 and 1800 - 112 * B == 8
    # eleven sharers copy the partially filled last prefix block; the twelfth
    # finds a reference count of one and writes in place
    assert wl.copy_pairs.shape == (11, 2)
    last_shared = wl.shared_blocks[112]
    assert np.all(wl.copy_pairs[:, 0] == last_shared)
    dsts = wl.copy_pairs[:, 1]
    assert len(set(dsts.tolist())) == 11 and last_shared not in dsts
    assert not set(dsts.tolist()) & set(wl.shared_blocks.tolist())
    for i in range(11):
        assert wl.block_tables[i, 112] == dsts[i]
    assert wl.block_tables[11, 112] == last_shared
    # full prefix blocks stay shared by every sequence
    for i in range(12):
        assert np.array_equal(wl.block_tables[i, :112], wl.shared_blocks[:112])
    used = _check_tables(wl)
    assert len(used) <= wl.num_blocks
    # no block other than the full prefix blocks is used by two sequences
    owners = {}
    for i in range(12):
        for p in wl.block_tables[i, 112:]:
            if p >= 0:
                assert int(p) not in owners
                owners[int(p)] = i


def test_block_pool_refcounts_and_free_list():
    pool = BlockPool(6, [3, 1, 4, 0, 5, 2])
    s = Sequence(pool, 4)
    assert s.reserve(5) == []
    assert s.table == [3, 1]
    t = s.fork()
    assert pool.ref[3] == 2 and pool.ref[1] == 2
    # writing into the shared partial block copies it first
    assert t.reserve(1) == [(1, 4)]
    assert t.table == [3, 4] and pool.ref[1] == 1 and pool.ref[4] == 1
    # the original writer now owns block 1 alone: no copy
    assert s.reserve(3) == []
    assert s.table == [3, 1]
    assert s.reserve(1) == []
    assert s.table == [3, 1, 0]
    t.release()
    assert pool.ref[3] == 1 and pool.ref[4] == 0 and 4 in pool.free
    with pytest.raises(ValueError):
        BlockPool(3, [0, 0, 1])


def test_nan_garbage_marks_only_unread_slots():
    wl = W.tiny(garbage="nan")
    mask = W.valid_slot_mask(wl)
    assert np.all(wl.k_cache[~mask] == W.NAN_BITS[W.F16])
    assert not np.any(wl.k_cache[mask] == W.NAN_BITS[W.F16])


def test_to_bits_round_to_nearest_even():
    # bfloat16: ties go to the even neighbour; binary16: numpy's conversion
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 65504.0], np.float32)
    bits = W.to_bits(x, W.BF16)
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x4780]
    assert np.array_equal(W.to_bits(x, W.F16), x.astype(np.float16).view(np.uint16))
