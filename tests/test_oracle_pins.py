"""Pins of the fp64 oracle to facts other than itself.

Each test checks the oracle against something the pages or mathematics fix:
worked examples printed on the pages (tests/golden/), closed forms, invariants,
a library routine for a special case, or a pure-Python brute force on tiny
inputs.  They are chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_worked_examples.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------- decoding

def test_f16_decode_matches_numpy_float16():
    # every binary16 pattern, against numpy's own binary16 -> float64 conversion
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_decode_matches_float32_upper_half():
    # bfloat16 is by definition the upper half of a binary32 pattern
    bits = np.arange(65536, dtype=np.uint32)
    ours = oracle.decode(bits.astype(np.uint16), oracle.BF16)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ---------------------------------------------------- addressing and blocks

def test_slot_formula_on_page_diagram(golden):
    g = golden["block_table_diagram"]
    for t, expected in g["token_slots"]:
        assert oracle.slot(g["block_table"], t, g["block_size"]) == expected


def test_blocks_for_closed_form_and_waste_bound():
    # ceil(T/B) blocks, fewer than B wasted slots per sequence
    for B in (1, 2, 4, 16, 32, 128):
        for T in range(0, 300):
            n = oracle.blocks_for(T, B)
            assert n == -(-T // B)
            assert 0 <= n * B - T < B


def test_slot_mapping_matches_block_walk():
    # brute force: walk the table block by block, slot by slot, and list the
    # physical slots in token order; the formula must give the same list
    rng = np.random.default_rng(3)
    B = 4
    table = rng.permutation(50)[:13].astype(np.int32)
    walked = []
    for p in table:
        for r in range(B):
            walked.append(int(p) * B + r)
    T = 49
    got = oracle.slot_mapping(table[None, :], np.zeros(T, np.int32), np.arange(T, dtype=np.int32), B)
    assert got.tolist() == walked[:T]


def test_cache_write_round_trip_and_untouched_rest():
    rng = np.random.default_rng(5)
    nb, B, H, D = 9, 4, 2, 8
    kc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    slots = np.array([5, -1, 17, 35, 0], dtype=np.int64)
    k = rng.integers(0, 65535, size=(5, H, D), dtype=np.uint16)
    v = rng.integers(0, 65535, size=(5, H, D), dtype=np.uint16)
    oracle.cache_write(kc, vc, k, v, slots)
    flat_k = kc.reshape(nb * B, H, D)
    flat_v = vc.reshape(nb * B, H, D)
    for i, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(flat_k[s], k[i]) and np.array_equal(flat_v[s], v[i])
    untouched = np.ones(nb * B, bool)
    untouched[[s for s in slots if s >= 0]] = False
    assert np.array_equal(flat_k[untouched], k0.reshape(nb * B, H, D)[untouched])
    assert np.array_equal(flat_v[untouched], v0.reshape(nb * B, H, D)[untouched])


def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(6)
    nb, B, H, D = 12, 4, 2, 8
    kc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[1, 7], [3, 8], [1, 9]], dtype=np.int32)
    oracle.copy_blocks(kc, vc, pairs)
    for s, d in pairs:
        assert np.array_equal(kc[d], k0[s]) and np.array_equal(vc[d], v0[s])
    rest = [b for b in range(nb) if b not in (7, 8, 9)]
    assert np.array_equal(kc[rest], k0[rest]) and np.array_equal(vc[rest], v0[rest])


def test_gather_bits_follows_table():
    rng = np.random.default_rng(7)
    nb, B, H, D = 10, 4, 3, 8
    kc = rng.integers(0, 65535, size=(nb, B, H, D), dtype=np.uint16)
    table = np.array([4, 0, 9], dtype=np.int32)
    T = 10
    g = oracle.gather_bits(kc, table, T)
    expected = np.concatenate([kc[4], kc[0], kc[9]], axis=0)[:T]
    assert np.array_equal(g, expected)


# ------------------------------------------------------------ attention math

def _brute_attention(q, K, V, scale):
    """Pure-Python loops with math.exp / math.fsum, the formula as printed."""
    T, D = len(K), len(q)
    s = [scale * math.fsum(q[d] * K[t][d] for d in range(D)) for t in range(T)]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = math.fsum(w)
    return [math.fsum(w[t] * V[t][d] for t in range(T)) / z for d in range(D)]


def test_attention_vs_pure_python_brute_force():
    rng = np.random.default_rng(11)
    for T, D in [(1, 4), (3, 8), (7, 16), (33, 8)]:
        q = rng.standard_normal(D)
        K = rng.standard_normal((T, D))
        V = rng.standard_normal((T, D))
        got = oracle.attention_1q(q, K, V, 1 / math.sqrt(D))
        ref = _brute_attention(q.tolist(), K.tolist(), V.tolist(), 1 / math.sqrt(D))
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_attention_vs_scipy_softmax():
    # special case of the textbook routine: softmax from scipy, matmul from numpy
    rng = np.random.default_rng(12)
    T, D = 257, 128
    q = rng.standard_normal(D)
    K = rng.standard_normal((T, D)) * 0.5
    V = rng.standard_normal((T, D)) * 0.5
    scale = 1 / math.sqrt(D)
    w = scipy.special.softmax(scale * (K @ q))
    np.testing.assert_allclose(oracle.attention_1q(q, K, V, scale), w @ V, rtol=1e-12, atol=1e-14)


def test_attention_closed_forms():
    rng = np.random.default_rng(13)
    D = 16
    V = rng.standard_normal((9, D))
    K = rng.standard_normal((9, D))
    q = rng.standard_normal(D)
    # T = 1: the output is the single value row
    assert np.array_equal(oracle.attention_1q(q, K[:1], V[:1], 0.25), V[0])
    # all keys equal: uniform weights, mean of V
    Keq = np.tile(K[:1], (9, 1))
    np.testing.assert_allclose(oracle.attention_1q(q, Keq, V, 0.25), V.mean(0), rtol=0, atol=1e-15)
    # zero query: uniform weights
    np.testing.assert_allclose(oracle.attention_1q(np.zeros(D), K, V, 0.25), V.mean(0), rtol=0,
                               atol=1e-15)
    # one overwhelming score: that value row
    Kbig = K.copy()
    Kbig[4] = q * 1e4
    np.testing.assert_allclose(oracle.attention_1q(q, Kbig, V, 1.0), V[4], rtol=0, atol=1e-12)


def test_attention_invariances():
    rng = np.random.default_rng(14)
    T, D = 40, 32
    q = rng.standard_normal(D)
    K = rng.standard_normal((T, D))
    V = rng.standard_normal((T, D))
    base = oracle.attention_1q(q, K, V, 0.3)
    # weights sum to one: shifting every value row by c shifts the output by c
    c = rng.standard_normal(D)
    np.testing.assert_allclose(oracle.attention_1q(q, K, V + c, 0.3), base + c, atol=1e-12)
    # the same score offset for every key leaves the output unchanged
    u = q / np.dot(q, q) * 7.0          # u.q = 7 for every key
    np.testing.assert_allclose(oracle.attention_1q(q, K + u, V, 0.3), base, atol=1e-12)
    # reordering keys together with their values leaves the output unchanged
    perm = rng.permutation(T)
    np.testing.assert_allclose(oracle.attention_1q(q, K[perm], V[perm], 0.3), base, atol=1e-13)
    # scale enters only through the product scale * q
    np.testing.assert_allclose(oracle.attention_1q(2 * q, K, V, 0.15), base, atol=1e-13)


def test_attention_spread_closed_forms():
    # spread_d = sum_t w_t |V_td - out_d| (the scale of the output error that
    # relative errors in the weights can cause; the GPU tests bound a kernel's
    # rounding of the weights by it)
    rng = np.random.default_rng(15)
    D = 16
    K = rng.standard_normal((9, D))
    V = rng.standard_normal((9, D))
    q = rng.standard_normal(D)
    # one token: the output is that row, with no deviation
    _, sp = oracle.attention_1q(q, K[:1], V[:1], 0.25, spread=True)
    assert np.array_equal(sp, np.zeros(D))
    # two tokens with equal weights (zero query): half their distance
    out, sp = oracle.attention_1q(np.zeros(D), K[:2], V[:2], 0.25, spread=True)
    np.testing.assert_allclose(sp, np.abs(V[0] - V[1]) / 2, rtol=1e-15, atol=0)
    # three equal weights on values 0, 1, 5: mean 2, deviations 2, 1, 3 -> 2
    V3 = np.array([[0.0], [1.0], [5.0]])
    out, sp = oracle.attention_1q(np.zeros(1), np.zeros((3, 1)), V3, 1.0, spread=True)
    assert out[0] == 2.0 and abs(sp[0] - 2.0) < 1e-15
    # weights 1/4, 3/4 (scores 0 and ln 3) on values 0 and 4: out 3, spread
    # 1/4 * 3 + 3/4 * 1 = 3/2
    K2 = np.array([[0.0], [math.log(3.0)]])
    out, sp = oracle.attention_1q(np.ones(1), K2, np.array([[0.0], [4.0]]), 1.0, spread=True)
    assert abs(out[0] - 3.0) < 1e-14 and abs(sp[0] - 1.5) < 1e-14
    # equal value rows: no deviation
    _, sp = oracle.attention_1q(q, K, np.tile(V[:1], (9, 1)), 0.25, spread=True)
    assert np.all(sp < 1e-15)


def test_attention_spread_invariances_and_perturbation_bound():
    rng = np.random.default_rng(16)
    T, D = 50, 24
    q = rng.standard_normal(D)
    K = rng.standard_normal((T, D))
    V = rng.standard_normal((T, D))
    out, sp = oracle.attention_1q(q, K, V, 0.4, spread=True)
    # a shift of every value row leaves it unchanged; a factor a scales it by |a|
    c = rng.standard_normal(D)
    np.testing.assert_allclose(oracle.attention_1q(q, K, V + c, 0.4, spread=True)[1], sp,
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(oracle.attention_1q(q, K, -3.0 * V, 0.4, spread=True)[1],
                               3.0 * sp, rtol=1e-12, atol=1e-13)
    # the property the GPU tests rely on: weights perturbed by relative
    # errors of at most u give a weighted mean within u * spread / (1 - u) of
    # the output; the worst signs (those of V - out) come close to it
    s = 0.4 * (K @ q)
    w = np.exp(s - s.max())
    w /= w.sum()
    u = 2.0 ** -8
    for trial in range(20):
        eps = rng.uniform(-u, u, (T, D)) if trial else u * np.sign(V - out)
        wp = w[:, None] * (1 + eps)
        moved = np.abs((wp * V).sum(0) / wp.sum(0) - out)
        assert np.all(moved <= u * sp / (1 - u) + 1e-15)
        if trial == 0:
            assert np.all(moved >= 0.99 * u * sp / (1 + u))


# --------------------------------------------------------- paged decode

def _bf16_bits(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _tiny_paged_case(rng, N=3, Hq=4, H_kv=2, D=8, B=4, nb=24, lens=(5, 1, 11)):
    q = _bf16_bits(rng.standard_normal((N, Hq, D)))
    kc = _bf16_bits(rng.standard_normal((nb, B, H_kv, D)))
    vc = _bf16_bits(rng.standard_normal((nb, B, H_kv, D)))
    perm = rng.permutation(nb).astype(np.int32)
    maxb = max(-(-T // B) for T in lens)
    bt = np.full((N, maxb), -1, np.int32)
    k = 0
    for i, T in enumerate(lens):
        n = -(-T // B)
        bt[i, :n] = perm[k:k + n]
        k += n
    return q, kc, vc, bt, np.array(lens, np.int32)


def test_paged_decode_vs_brute_force_through_table():
    # brute force on tiny inputs: follow the table token by token in Python,
    # decode the bf16 patterns through float32, then the printed formula
    rng = np.random.default_rng(21)
    q, kc, vc, bt, sl = _tiny_paged_case(rng)
    N, Hq, D = q.shape
    B, H_kv = kc.shape[1], kc.shape[2]
    G = Hq // H_kv
    scale = 1 / math.sqrt(D)
    got = oracle.paged_decode(q, kc, vc, oracle.BF16, bt, sl, scale)
    f = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for i in range(N):
        for hq in range(Hq):
            h = hq // G
            Ks, Vs = [], []
            for t in range(int(sl[i])):
                p = bt[i][t // B]
                Ks.append(f(kc[p, t % B, h]).tolist())
                Vs.append(f(vc[p, t % B, h]).tolist())
            ref = _brute_attention(f(q[i, hq]).tolist(), Ks, Vs, scale)
            np.testing.assert_allclose(got[i, hq], ref, rtol=1e-13, atol=1e-14)


def test_paged_equals_contiguous_with_identity_table():
    rng = np.random.default_rng(22)
    T, H_kv, Hq, D, B = 37, 2, 6, 16, 8
    nb = -(-T // B)
    kc = _bf16_bits(rng.standard_normal((nb, B, H_kv, D)))
    vc = _bf16_bits(rng.standard_normal((nb, B, H_kv, D)))
    q = _bf16_bits(rng.standard_normal((1, Hq, D)))
    bt = np.arange(nb, dtype=np.int32)[None, :]
    paged = oracle.paged_decode(q, kc, vc, oracle.BF16, bt, np.array([T], np.int32), 0.25)[0]
    Kc = oracle.decode(kc, oracle.BF16).reshape(nb * B, H_kv, D)[:T]
    Vc = oracle.decode(vc, oracle.BF16).reshape(nb * B, H_kv, D)[:T]
    cont = oracle.contiguous_decode(oracle.decode(q[0], oracle.BF16), Kc, Vc, 0.25)
    assert np.array_equal(paged, cont)


def test_paged_decode_invariant_under_block_placement():
    # the same logical cache placed in two different physical arrangements
    rng = np.random.default_rng(23)
    N, Hq, H_kv, D, B, nb = 2, 4, 2, 8, 4, 20
    lens = np.array([13, 6], np.int32)
    q = _bf16_bits(rng.standard_normal((N, Hq, D)))
    logical_k = [_bf16_bits(rng.standard_normal((-(-T // B), B, H_kv, D))) for T in lens]
    logical_v = [_bf16_bits(rng.standard_normal((-(-T // B), B, H_kv, D))) for T in lens]
    outs = []
    for seed in (0, 1):
        perm = np.random.default_rng(seed).permutation(nb).astype(np.int32)
        kc = np.zeros((nb, B, H_kv, D), np.uint16)
        vc = np.zeros((nb, B, H_kv, D), np.uint16)
        bt = np.full((N, 4), -1, np.int32)
        k = 0
        for i in range(N):
            for j in range(logical_k[i].shape[0]):
                p = perm[k]
                k += 1
                bt[i, j] = p
                kc[p] = logical_k[i][j]
                vc[p] = logical_v[i][j]
        outs.append(oracle.paged_decode(q, kc, vc, oracle.BF16, bt, lens, 0.3))
    assert np.array_equal(outs[0], outs[1])


def test_gqa_equals_replicated_heads():
    # G query heads per KV head == the same cache with each KV head repeated G
    # times (contiguous groups: query head hq reads KV head hq // G)
    rng = np.random.default_rng(24)
    N, Hq, H_kv, D, B, nb = 2, 8, 2, 8, 4, 16
    G = Hq // H_kv
    q, kc, vc, bt, sl = _tiny_paged_case(rng, N=N, Hq=Hq, H_kv=H_kv, D=D, B=B, nb=nb, lens=(9, 14))
    gqa = oracle.paged_decode(q, kc, vc, oracle.BF16, bt, sl, 0.35)
    kc_rep = np.ascontiguousarray(np.repeat(kc, G, axis=2))
    vc_rep = np.ascontiguousarray(np.repeat(vc, G, axis=2))
    mha = oracle.paged_decode(q, kc_rep, vc_rep, oracle.BF16, bt, sl, 0.35)
    assert np.array_equal(gqa, mha)


def test_paged_decode_ignores_unused_slots():
    # slots past seq_len in the last block (and blocks past ceil(T/B) in the
    # table) hold garbage, NaN included; the result must not change
    rng = np.random.default_rng(25)
    q, kc, vc, bt, sl = _tiny_paged_case(rng)
    base = oracle.paged_decode(q, kc, vc, oracle.BF16, bt, sl, 0.3)
    kc2, vc2 = kc.copy(), vc.copy()
    B = kc.shape[1]
    used = np.zeros((kc.shape[0], B), bool)
    for i, T in enumerate(sl):
        for t in range(int(T)):
            used[bt[i, t // B], t % B] = True
    kc2[~used] = 0x7FC0
    vc2[~used] = 0x7FC0
    assert np.array_equal(oracle.paged_decode(q, kc2, vc2, oracle.BF16, bt, sl, 0.3), base)


def test_zero_length_sequence_gives_zero_row():
    rng = np.random.default_rng(26)
    q, kc, vc, bt, sl = _tiny_paged_case(rng)
    sl = sl.copy()
    sl[1] = 0
    out = oracle.paged_decode(q, kc, vc, oracle.BF16, bt, sl, 0.3)
    assert np.all(out[1] == 0)


# ------------------------------------------- capacity arithmetic (the pages)

def test_static_batch_fraction(golden):
    g = golden["static_batch"]
    num, den = oracle.static_batch_useful_fraction(g["prompts"], g["outputs"])
    assert (num, den) == (g["numerator"], g["denominator"])
    assert round(100 * num / den) == g["percent_rounded"]


def test_fragmentation_example(golden):
    g = golden["fragmentation"]
    L = g["lengths"]
    reserved = len(L) * g["max_len"]
    assert reserved == g["contiguous_reserved_slots"]
    assert reserved - oracle.wasted_slots_contiguous(L, g["max_len"]) == g["tokens"]
    assert oracle.allocated_slots_paged(L, g["block_size"]) == g["paged_allocated_slots"]
    assert oracle.wasted_slots_paged(L, g["block_size"]) == g["paged_allocated_slots"] - g["tokens"]
    assert oracle.wasted_slots_paged(L, g["block_size"]) < len(L) * g["block_size"]
    assert round(100 * g["tokens"] / reserved) == g["contiguous_used_percent_rounded"]
    assert round(100 * g["tokens"] / g["paged_allocated_slots"]) == g["paged_used_percent_rounded"]


def test_pool_sizing_example(golden):
    g = golden["pool_sizing"]
    bb = oracle.block_bytes(g["layers"], g["block_size"], g["kv_heads"], g["head_dim"],
                            g["dtype_bytes"])
    assert bb == g["block_bytes"] == 8 * 2**20
    nblocks = oracle.pool_blocks(g["pool_gib"] * 2**30, bb)
    assert abs(nblocks - g["num_blocks_approx"]) / g["num_blocks_approx"] < 0.01
    tokens = nblocks * g["block_size"]
    assert abs(tokens - g["tokens_approx"]) / g["tokens_approx"] < 0.01
    assert tokens // 4096 == g["requests_at_4096_tokens"]
    assert abs(tokens // 512 - g["requests_at_512_tokens_approx"]) <= 5


def test_kv_bytes_per_token(golden):
    g = golden["kv_bytes_per_token"]
    for m in g["models"]:
        assert oracle.kv_bytes_per_token(m["layers"], m["kv_heads"], m["head_dim"],
                                         m["dtype_bytes"]) == m["bytes_per_token"]
    qwen = g["models"][0]
    per = oracle.kv_bytes_per_token(qwen["layers"], qwen["kv_heads"], qwen["head_dim"], 2)
    for tokens, measured in g["qwen2_measured"]:
        assert per * tokens == measured
    assert 131072 * 4096 == g["llama3_4096_tokens_mib"] * 2**20
    assert 524288 * 4096 == g["llama2_4096_tokens_mib"] * 2**20


def test_capacity_example(golden):
    g = golden["capacity"]
    per_tok = g["bytes_per_token"]
    reserve = per_tok * g["reserve_tokens"]
    assert round(reserve / 1e6) == g["reserve_mb"]
    free = g["free_gb"] * 1e9
    assert oracle.requests_that_fit(free, reserve) == g["contiguous_requests"]
    assert round(100 * (1 - g["typical_tokens"] / g["reserve_tokens"]), 1) == g["untouched_percent"]
    nblk = oracle.blocks_for(g["typical_tokens"], 16)
    assert nblk == g["blocks_per_typical_request"]
    paged = nblk * 16 * per_tok
    assert round(paged / 1e6, 1) == g["paged_request_mb"]
    assert oracle.requests_that_fit(free, paged) == g["paged_requests"]
    assert round(g["paged_requests"] / g["contiguous_requests"], 1) == g["gain"]
    separate = g["shared_prefix_requests"] * g["shared_prefix_tokens"] * per_tok
    shared = g["shared_prefix_tokens"] * per_tok
    assert round(separate / 1e9, 2) == g["separate_copies_gb"]
    assert round(shared / 1e9, 3) == g["shared_gb"]
    assert round((separate - shared) / 1e9, 2) == g["freed_gb"]
    assert oracle.requests_that_fit(separate - shared, paged) == g["extra_requests"]


def test_sliding_window_bound(golden):
    g = golden["sliding_window"]
    assert oracle.sliding_window_max_blocks(g["window"], g["block_size"]) == g["max_blocks"]


def test_swap_blocks_moves_whole_blocks_and_round_trips():
    # "Swapping moves physical blocks from the GPU memory to the CPU's system
    # memory ... the engine swaps the blocks back": a block swapped out and
    # back into another block holds the same bits, and the decode through a
    # table that points at the new blocks does not change
    wl = W.random_workload(61, W.BF16, 8, 2, 64, 16, [40, 70], num_blocks=20)
    host_k = np.zeros((10,) + wl.k_cache.shape[1:], np.uint16)
    host_v = np.zeros_like(host_k)
    used = np.unique(wl.block_tables[wl.block_tables >= 0])
    out_pairs = np.stack([used, np.arange(used.size)], axis=1)
    oracle.swap_blocks(wl.k_cache, wl.v_cache, host_k, host_v, out_pairs)
    assert np.array_equal(host_k[:used.size], wl.k_cache[used])
    assert np.array_equal(host_v[:used.size], wl.v_cache[used])
    assert not host_k[used.size:].any()
    kc = np.zeros_like(wl.k_cache)
    vc = np.zeros_like(wl.v_cache)
    free = np.setdiff1d(np.arange(wl.num_blocks), used)[::-1][:used.size]
    oracle.swap_blocks(host_k, host_v, kc, vc, np.stack([np.arange(used.size), free], axis=1))
    remap = dict(zip(used.tolist(), free.tolist()))
    bt = np.vectorize(lambda b: remap.get(int(b), -1))(wl.block_tables).astype(np.int32)
    a = oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                            wl.seq_lens, wl.scale)
    b = oracle.paged_decode(wl.q, kc, vc, wl.dtype, bt, wl.seq_lens, wl.scale)
    assert np.array_equal(a, b)
