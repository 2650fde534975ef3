"""Pins of the oracle's sliding-window decode ("vLLM Framework and Inference
Engine Design", section "How does it support prompts of arbitrary length? Does
it have a sliding window?": each token attends only to the last W tokens; the
blocks before the window can be released; at most ceil(W/B) + 1 blocks per
sequence).  Reading: the query of position T - 1 attends to [max(0, T - W), T).
"""
import numpy as np

import oracle
import workloads as W


def _decode_w(wl, window, bt=None):
    return oracle.paged_decode_window(wl.q, wl.k_cache, wl.v_cache, wl.dtype,
                                      wl.block_tables if bt is None else bt, wl.seq_lens, window,
                                      wl.scale)


def test_window_no_shorter_than_the_context_is_full_attention():
    wl = W.random_workload(81, W.BF16, 8, 2, 64, 16, [1, 15, 16, 17, 100, 257])
    full = oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                               wl.seq_lens, wl.scale)
    assert np.array_equal(_decode_w(wl, 257), full)
    assert np.array_equal(_decode_w(wl, 10 ** 6), full)
    assert np.array_equal(_decode_w(wl, 0), full)


def test_window_of_one_token_returns_its_value_row():
    wl = W.random_workload(82, W.F16, 6, 3, 128, 8, [1, 9, 33, 64])
    out = _decode_w(wl, 1)
    G = wl.group
    for i, T in enumerate(wl.seq_lens):
        for h in range(wl.num_kv_heads):
            vt = oracle.gather_head(wl.v_cache, wl.dtype, wl.block_tables[i], int(T), h)[-1]
            for g in range(G):
                assert np.array_equal(out[i, h * G + g], vt)


def test_window_equals_contiguous_attention_over_the_last_w_tokens():
    wl = W.random_workload(83, W.BF16, 8, 2, 64, 16, [40, 100, 300])
    for window in (1, 15, 16, 17, 50, 299):
        out = _decode_w(wl, window)
        for i, T in enumerate(wl.seq_lens):
            T = int(T)
            s0 = max(0, T - window)
            K = np.stack([oracle.gather_head(wl.k_cache, wl.dtype, wl.block_tables[i], T, h)
                          for h in range(wl.num_kv_heads)], axis=1)[s0:]
            V = np.stack([oracle.gather_head(wl.v_cache, wl.dtype, wl.block_tables[i], T, h)
                          for h in range(wl.num_kv_heads)], axis=1)[s0:]
            q = oracle.decode(wl.q[i], wl.dtype)
            ref = oracle.contiguous_decode(q, K, V, wl.scale)
            np.testing.assert_allclose(out[i], ref, rtol=1e-13, atol=1e-15)


def test_released_table_entries_are_never_read():
    wl = W.random_workload(84, W.BF16, 4, 2, 64, 16, [200, 700, 33], window=100)
    bt = wl.block_tables.copy()
    assert np.any(bt < 0)                      # blocks before the window were released
    a = _decode_w(wl, 100)
    bt2 = bt.copy()
    bt2[bt2 < 0] = bt[0, -1] if bt[0, -1] >= 0 else int(bt[bt >= 0][0])   # a valid, wrong block
    b = _decode_w(wl, 100, bt2)
    assert np.array_equal(a, b)


def test_sliding_window_workload_keeps_at_most_the_pages_block_bound():
    wl = W.mistral_7b_swa(num_seqs=6, num_blocks=2_000)
    bound = oracle.sliding_window_max_blocks(wl.window, wl.block_size)
    assert bound == 257
    live = (wl.block_tables >= 0).sum(axis=1)
    assert np.all(live <= bound)
    assert np.all(wl.seq_lens > wl.window)
    # the live blocks are exactly those reaching into the window
    for i, T in enumerate(wl.seq_lens):
        first = (int(T) - wl.window) // wl.block_size
        assert np.all(wl.block_tables[i, :first] == -1)
        assert np.all(wl.block_tables[i, first:-(-int(T) // wl.block_size)] >= 0)
