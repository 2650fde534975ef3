"""Pins of the oracle's multi-query paged attention (chunked prefill;
"vLLM Framework and Inference Engine Design", section "How does it support
prompts of arbitrary length?": long prompts are processed in chunks that run in
one batch with other requests' decode tokens).  Reading: a sequence's L new
tokens sit at the end of its T cached tokens (written before attention); new
token j, at position T - L + j, attends causally to tokens [0, T - L + j].
"""
import numpy as np
import scipy.special

import oracle
import workloads as W


def test_single_token_steps_are_the_decode():
    wl = W.random_prefill(121, W.BF16, 8, 2, 64, 16, [0, 15, 16, 200], [1, 1, 1, 1])
    got = oracle.paged_prefill(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                               wl.seq_lens, wl.query_start, wl.scale)
    ref = oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                              wl.seq_lens, wl.scale)
    assert np.array_equal(got, ref)


def test_chunk_equals_dense_causal_softmax_attention():
    # the textbook masked softmax attention (scipy's softmax over scores with
    # -inf above the diagonal), on the contiguous gathered cache
    wl = W.random_prefill(122, W.F16, 6, 3, 64, 8, [0, 7, 40], [33, 9, 64])
    got = oracle.paged_prefill(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                               wl.seq_lens, wl.query_start, wl.scale)
    G = wl.group
    for i, T in enumerate(wl.seq_lens):
        T = int(T)
        q0, q1 = wl.query_start[i], wl.query_start[i + 1]
        L = q1 - q0
        pos = np.arange(T - L, T)
        for h in range(wl.num_kv_heads):
            K = oracle.gather_head(wl.k_cache, wl.dtype, wl.block_tables[i], T, h)
            V = oracle.gather_head(wl.v_cache, wl.dtype, wl.block_tables[i], T, h)
            for g in range(G):
                Q = oracle.decode(wl.q[q0:q1, h * G + g], wl.dtype)
                S = wl.scale * (Q @ K.T)
                S[np.arange(T)[None, :] > pos[:, None]] = -np.inf
                ref = scipy.special.softmax(S, axis=1) @ V
                np.testing.assert_allclose(got[q0:q1, h * G + g], ref, rtol=1e-12, atol=1e-14)


def test_splitting_a_prompt_into_chunks_changes_nothing():
    # one 100-token chunk vs the same prompt as chunks of 30, 50 and 20 tokens,
    # each attending to what the previous chunks left in the cache
    wl = W.random_prefill(123, W.BF16, 4, 2, 128, 16, [20], [100])
    whole = oracle.paged_prefill(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                                 wl.seq_lens, wl.query_start, wl.scale)
    done = 0
    for c in (30, 50, 20):
        T = 20 + done + c
        part = oracle.paged_prefill(wl.q[done:done + c], wl.k_cache, wl.v_cache, wl.dtype,
                                    wl.block_tables, np.array([T], np.int32),
                                    np.array([0, c], np.int32), wl.scale)
        assert np.array_equal(part, whole[done:done + c])
        done += c


def test_first_token_of_an_empty_prefix_returns_its_own_value_row():
    wl = W.random_prefill(124, W.F16, 4, 4, 64, 16, [0], [5])
    got = oracle.paged_prefill(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                               wl.seq_lens, wl.query_start, wl.scale)
    for h in range(4):
        v0 = oracle.gather_head(wl.v_cache, wl.dtype, wl.block_tables[0], 1, h)[0]
        assert np.array_equal(got[0, h], v0)
