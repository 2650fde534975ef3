"""Pins of the oracle's FP8 (E4M3) KV-cache arithmetic, each checked against
something other than the oracle itself: the E4M3 value set rebuilt from the
binary16 number line, torch's own float8_e4m3fn conversion, a brute-force
nearest-value search, and the already pinned 16-bit decode on inputs where the
two must agree exactly.

Reading (the pages name only "fp8" and its halved memory; "vLLM Framework and
Inference Engine Design", section "How can one customize the tokenizer, cache
strategy, or scheduler strategy?"): OCP E4M3, one scale per tensor, code =
e4m3_rne_satfinite(float32(x) / scale), value = e4m3(code) * scale.
"""
import numpy as np
import pytest

import oracle
import workloads as W

CODES = np.arange(256, dtype=np.uint8)
FINITE = CODES[(CODES & 0x7F) != 0x7F]


def _e4m3_values_from_binary16():
    # every binary16 value that E4M3 can hold: magnitude at most 448 and a
    # multiple of the E4M3 spacing at its binade (2^-9 below 2^-6)
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    h = h[np.isfinite(h)]
    a = np.abs(h)
    ok = a <= 448.0
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    spacing = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    ok &= np.mod(a, spacing) == 0
    return np.unique(h[ok])


def test_e4m3_value_set_matches_the_binary16_derivation():
    vals = oracle.e4m3_decode(FINITE)
    assert np.all(np.isfinite(vals))
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    assert FINITE.size == 254
    assert np.array_equal(np.unique(vals), _e4m3_values_from_binary16())
    # codes 0x00..0x7E increase strictly; the sign bit mirrors them
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9 and pos[8] == 2.0 ** -6
    assert oracle.e4m3_decode(np.array([0x38], np.uint8))[0] == 1.0


def test_e4m3_round_trip_of_every_finite_code():
    vals = oracle.e4m3_decode(FINITE).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), FINITE)


def _nearest_even(x, codes, vals):
    """Brute force: the finite code nearest to x, ties to an even fraction LSB,
    beyond the largest magnitude the largest code of that sign."""
    out = np.empty(x.shape, np.uint8)
    for n, xv in enumerate(x.astype(np.float64)):
        d = np.abs(vals - xv)
        best = np.flatnonzero(d == d.min())
        if best.size > 1:
            even = best[(codes[best] & 1) == 0]
            best = even if even.size else best
        c = codes[best]
        # signed zero follows the sign of x
        if vals[best[0]] == 0.0:
            c = np.array([0x80 if np.signbit(xv) else 0x00])
        out[n] = c[0]
    return out


def test_e4m3_encoder_against_brute_force_nearest():
    rng = np.random.default_rng(7)
    vals = oracle.e4m3_decode(FINITE)
    # random magnitudes over the whole range, exact midpoints, and the edges
    x = (rng.standard_normal(3000) * np.exp2(rng.integers(-12, 9, 3000))).astype(np.float32)
    pos = np.sort(np.unique(vals[vals >= 0]))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    edges = np.array([0.0, -0.0, 2.0 ** -10, 2.0 ** -9 * 1.5, 447.9, 448.0, 463.9, -447.0],
                     np.float32)
    x = np.concatenate([x, mids, -mids, edges])
    x = x[np.abs(x) <= 448]
    assert np.array_equal(oracle.e4m3_encode(x), _nearest_even(x, FINITE, vals))


def test_e4m3_saturates_beyond_the_largest_magnitude():
    x = np.array([448.5, 464.0, 1e6, np.inf, -500.0, -np.inf], np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e4m3_agrees_with_torch_float8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    vals = oracle.e4m3_decode(FINITE)
    t = torch.from_numpy(FINITE.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(t, vals)
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-11, 8, 20000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    mine = oracle.e4m3_encode(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, theirs)


def test_fp8_cache_write_stores_the_quantized_rows_at_their_slots():
    wl = W.random_workload(41, W.BF16, 4, 2, 64, 8, [5, 17, 30])
    kc = np.full(wl.k_cache.shape, 0x7F, np.uint8)   # NaN codes everywhere
    vc = kc.copy()
    slots = oracle.slot_mapping(wl.block_tables, wl.new_seq, wl.new_pos, wl.block_size)
    ks, vs = 0.037, 0.21
    oracle.cache_write_fp8(kc, vc, wl.k_new, wl.v_new, wl.dtype, slots, ks, vs)
    H, D = kc.shape[2], kc.shape[3]
    kf = kc.reshape(-1, H, D)
    vf = vc.reshape(-1, H, D)
    kx = oracle.decode(wl.k_new, wl.dtype).astype(np.float32)
    vx = oracle.decode(wl.v_new, wl.dtype).astype(np.float32)
    for n, s in enumerate(slots):
        assert np.array_equal(kf[s], oracle.e4m3_encode(kx[n] / np.float32(ks)))
        assert np.array_equal(vf[s], oracle.e4m3_encode(vx[n] / np.float32(vs)))
    written = np.zeros(kf.shape[0], bool)
    written[slots] = True
    assert np.all(kf[~written] == 0x7F) and np.all(vf[~written] == 0x7F)


def test_fp8_decode_equals_the_16bit_decode_of_the_same_values():
    # with power-of-two scales every dequantized value is a binary16 value, so
    # the fp8 decode must equal the (pinned) 16-bit decode exactly
    rng = np.random.default_rng(9)
    wl = W.random_workload(42, W.F16, 8, 2, 64, 16, [1, 16, 40, 200])
    kc = W.random_e4m3_codes(rng, wl.k_cache.shape)
    vc = W.random_e4m3_codes(rng, wl.v_cache.shape)
    ks, vs = 0.5, 0.125
    got = oracle.paged_decode_fp8(wl.q, kc, vc, W.F16, ks, vs, wl.block_tables, wl.seq_lens,
                                  wl.scale)
    k16 = (oracle.e4m3_decode(kc) * ks).astype(np.float16).view(np.uint16)
    v16 = (oracle.e4m3_decode(vc) * vs).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.decode(k16, W.F16), oracle.e4m3_decode(kc) * ks)
    ref = oracle.paged_decode(wl.q, k16, v16, W.F16, wl.block_tables, wl.seq_lens, wl.scale)
    assert np.array_equal(got, ref)


def test_fp8_decode_scales_linearly_in_the_value_scale():
    rng = np.random.default_rng(10)
    wl = W.random_workload(43, W.BF16, 4, 4, 128, 16, [33, 90])
    kc = W.random_e4m3_codes(rng, wl.k_cache.shape)
    vc = W.random_e4m3_codes(rng, wl.v_cache.shape)
    a = oracle.paged_decode_fp8(wl.q, kc, vc, W.BF16, 0.02, 0.25, wl.block_tables, wl.seq_lens,
                                wl.scale)
    b = oracle.paged_decode_fp8(wl.q, kc, vc, W.BF16, 0.02, 1.0, wl.block_tables, wl.seq_lens,
                                wl.scale)
    assert np.array_equal(a * 4, b)
