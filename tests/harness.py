"""Test harness: one step of the paged decode path through the CUDA library
(C ABI, via the binding) and the same step through the fp64 oracle, on the
same seeded workload.

A step is: copy-on-write block copies (if any), slot mapping, cache write,
decode ("vLLM Framework and Inference Engine Design": K/V are written to their
slots when computed; the query of the newest token then attends over
seq_len tokens, its own included).
"""
import json
import os

import numpy as np
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W

# decode tolerance per element: |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL = 4e-3
RTOL = 1e-2

TORCH_DTYPE = {W.F16: torch.float16, W.BF16: torch.bfloat16}


def to_dev(bits, dtype, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DTYPE[dtype])


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class GpuState:
    """The workload's inputs resident on the GPU."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        if wl.fp8:   # uint8 E4M3 codes
            self.k_cache = torch.from_numpy(wl.k_cache).to(device)
            self.v_cache = torch.from_numpy(wl.v_cache).to(device)
        else:
            self.k_cache = to_dev(wl.k_cache, wl.dtype, device)
            self.v_cache = to_dev(wl.v_cache, wl.dtype, device)
        self.q = to_dev(wl.q, wl.dtype, device)
        self.k_new = to_dev(wl.k_new, wl.dtype, device)
        self.v_new = to_dev(wl.v_new, wl.dtype, device)
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        self.new_seq = torch.from_numpy(wl.new_seq).to(device)
        self.new_pos = torch.from_numpy(wl.new_pos).to(device)
        self.pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, np.int32)).to(device)
        self.query_start = (None if wl.query_start is None
                            else torch.from_numpy(wl.query_start).to(device))
        self.err = torch.zeros(1, dtype=torch.int32, device=device)


def gpu_step(st, flags=pa.PA_DECODE_AUTO, num_ctas=0, decode=True):
    """Runs the step; returns (out tensor or None, slot_mapping tensor)."""
    wl = st.wl
    if st.pairs.numel():
        pa.pa_copy_blocks(st.pairs, st.k_cache, st.v_cache, err=st.err)
    slots = pa.pa_slot_mapping(st.block_tables, st.new_seq, st.new_pos, wl.block_size,
                               wl.num_blocks, err=st.err)
    if wl.fp8:
        pa.pa_cache_write_fp8(st.k_new, st.v_new, slots, st.k_cache, st.v_cache, wl.k_scale,
                              wl.v_scale, err=st.err)
    else:
        pa.pa_cache_write(st.k_new, st.v_new, slots, st.k_cache, st.v_cache, err=st.err)
    out = None
    if decode:
        out = gpu_decode(st, st.seq_lens, flags=flags, num_ctas=num_ctas)
    return out, slots


def gpu_decode(st, seq_lens, flags=pa.PA_DECODE_AUTO, num_ctas=0, workspace=None):
    """The decode call of the workload's cache type."""
    wl = st.wl
    if wl.query_start is not None:
        return pa.pa_prefill(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens,
                             st.query_start, wl.scale, workspace=workspace, err=st.err)
    if wl.window > 0:
        return pa.pa_decode_window(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens,
                                   wl.scale, wl.window, flags=flags, num_ctas=num_ctas,
                                   workspace=workspace, err=st.err)
    if wl.fp8:
        return pa.pa_decode_fp8(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens,
                                wl.scale, wl.k_scale, wl.v_scale, flags=flags,
                                num_ctas=num_ctas, workspace=workspace, err=st.err)
    return pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens, wl.scale,
                        flags=flags, num_ctas=num_ctas, workspace=workspace, err=st.err)


class OracleState:
    """Host copies of the workload's pools, stepped by the oracle."""

    def __init__(self, wl):
        self.wl = wl
        self.k_cache = wl.k_cache.copy()
        self.v_cache = wl.v_cache.copy()

    def step(self):
        wl = self.wl
        if wl.copy_pairs.size:
            oracle.copy_blocks(self.k_cache, self.v_cache, wl.copy_pairs)
        self.slots = oracle.slot_mapping(wl.block_tables, wl.new_seq, wl.new_pos, wl.block_size)
        if wl.fp8:
            oracle.cache_write_fp8(self.k_cache, self.v_cache, wl.k_new, wl.v_new, wl.dtype,
                                   self.slots, wl.k_scale, wl.v_scale)
        else:
            oracle.cache_write(self.k_cache, self.v_cache, wl.k_new, wl.v_new, self.slots)

    def decode(self, seq_ids=None, threads=0, seq_lens=None, spread=False):
        """The oracle's output for the step; with spread=True, (out, spread)."""
        wl = self.wl
        sl = wl.seq_lens if seq_lens is None else seq_lens
        if wl.query_start is not None:
            return oracle.paged_prefill(wl.q, self.k_cache, self.v_cache, wl.dtype,
                                        wl.block_tables, sl, wl.query_start, wl.scale,
                                        threads=threads, spread=spread)
        if wl.window > 0:
            return oracle.paged_decode_window(wl.q, self.k_cache, self.v_cache, wl.dtype,
                                              wl.block_tables, sl, wl.window, wl.scale,
                                              seq_ids=seq_ids, threads=threads, spread=spread)
        if wl.fp8:
            return oracle.paged_decode_fp8(wl.q, self.k_cache, self.v_cache, wl.dtype, wl.k_scale,
                                           wl.v_scale, wl.block_tables, sl, wl.scale,
                                           seq_ids=seq_ids, threads=threads, spread=spread)
        return oracle.paged_decode(wl.q, self.k_cache, self.v_cache, wl.dtype, wl.block_tables,
                                   sl, wl.scale, seq_ids=seq_ids, threads=threads, spread=spread)


def gpu_out_f64(out):
    return out.float().cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------------------
# Rounding diagnostics against the oracle rounded once to the output dtype
# ---------------------------------------------------------------------------

def unit_roundoff(dtype):
    """Largest relative error of one round-to-nearest-even into dtype."""
    return 2.0 ** -8 if dtype == W.BF16 else 2.0 ** -11


def weight_roundoff(wl, flags=0):
    """Relative rounding of the softmax weights P on the path that runs wl.
    The CUDA-core decode (group size 1 unless the tensor-core kernel is
    forced) keeps P in fp32.  The 16-bit tensor-core decode feeds P to its
    P.V products as a pair hi = round(P), lo = round(P - hi) of 16-bit values,
    whose sum carries P to within 2^-16 (bfloat16) or 2^-22 (binary16); 2^-15
    bounds both.  The E4M3 decode feeds binary16 P (2^-11), the prefill P in
    the model dtype."""
    G = wl.num_q_heads // wl.num_kv_heads
    if wl.query_start is not None:
        return unit_roundoff(wl.dtype)
    mma = (flags & 0xff) == pa.PA_DECODE_MMA or ((flags & 0xff) == pa.PA_DECODE_AUTO and G > 1)
    if not mma:
        return 0.0
    return 2.0 ** -11 if wl.fp8 else 2.0 ** -15


def _f64_to_f32_round_to_odd(x):
    """binary32 bit patterns of x rounded to odd (truncate, then set the last
    bit if inexact): rounding that once more to fewer bits gives the correctly
    rounded result, with no double-rounding error."""
    x = np.asarray(x, np.float64)
    f = x.astype(np.float32)
    u = f.view(np.uint32).astype(np.int64)
    back = f.astype(np.float64)
    toward_zero_fix = np.abs(back) > np.abs(x)
    u = np.where(toward_zero_fix, u - 1, u)
    inexact = f.astype(np.float64) != x
    u = np.where(inexact, u | 1, u)
    return u.astype(np.uint32)


def round_bits(x, dtype):
    """fp64 values -> 16-bit patterns of dtype, round to nearest even."""
    x = np.asarray(x, np.float64)
    if dtype == W.F16:
        return x.astype(np.float16).view(np.uint16)   # numpy rounds fp64 -> binary16 once
    u = _f64_to_f32_round_to_odd(x).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bits_to_f64(bits, dtype):
    bits = np.asarray(bits, np.uint16)
    if dtype == W.F16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ordered(bits):
    """16-bit sign-magnitude patterns -> integers in value order (+0 = -0)."""
    b = np.asarray(bits, np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_spacing(bits, dtype):
    """Spacing of dtype's values just above |value| of each pattern."""
    v = np.abs(bits_to_f64(bits, dtype))
    if dtype == W.F16:
        return np.spacing(v.astype(np.float16)).astype(np.float64)
    return np.spacing(v.astype(np.float32)).astype(np.float64) * 65536.0


# fp32 work of the kernels (score products, exp2, running sums, merges) is
# budgeted at 2^-14 of |o| + spread: 2^10 times binary32's unit roundoff,
# ample for sums over up to 2^20 terms whose errors add like a random walk
FP32_SLACK = 2.0 ** -14


def rounding_report(got_bits, ref, spread, dtype, u_p, what=""):
    """Compares kernel output patterns with the oracle.

    The kernel's result x (fp32, before its one rounding) is a weighted mean
    of the value rows whose weights were rounded by at most u_p relatively,
    so |x - o| <= u_p * spread (1 + 2^-6) + fp32 terms, and the output
    rounding adds at most half the spacing at the result:
        |g - o| <= ulp(g) / 2 + u_p * spread * (1 + 2^-6) + 2^-14 (|o| + spread).
    With u_p = 0 and small fp32 terms this says g is within one ulp of the
    oracle rounded once to dtype.  Returns the figures of the comparison and
    raises AssertionError on an element past the bound."""
    g_bits = np.asarray(got_bits, np.uint16).reshape(-1)
    o = np.asarray(ref, np.float64).reshape(-1)
    sp = np.asarray(spread, np.float64).reshape(-1)
    assert g_bits.size == o.size == sp.size
    g = bits_to_f64(g_bits, dtype)
    assert np.all(np.isfinite(g)), "%s: non-finite output" % what
    err = np.abs(g - o)
    bound = (0.5 * ulp_spacing(g_bits, dtype) + u_p * sp * (1 + 2.0 ** -6)
             + FP32_SLACK * (np.abs(o) + sp))
    ulps = np.abs(_ordered(g_bits) - _ordered(round_bits(o, dtype)))
    big = np.abs(o) >= 1e-3
    rep = {
        "what": what, "n": int(o.size), "u_p": u_p,
        "frac_0ulp": float(np.mean(ulps == 0)), "frac_le1ulp": float(np.mean(ulps <= 1)),
        "max_ulp": int(ulps.max()) if ulps.size else 0,
        "max_ulp_o_ge_1e-3": int(ulps[big].max()) if big.any() else 0,
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_abs_o_ge_1e-3": float(err[big].max()) if big.any() else 0.0,
        "max_rel_o_ge_1e-3": float((err[big] / np.abs(o[big])).max()) if big.any() else 0.0,
        "bound_use": float((err / bound).max()) if err.size else 0.0,
    }
    path = os.environ.get("PA_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rep) + "\n")
    bad = err > bound
    if bad.any():
        idx = np.flatnonzero(bad)[:5].tolist()
        raise AssertionError("%s: %d of %d elements past the rounding bound (worst %.3g of the "
                             "bound); flat indices %s" % (what, int(bad.sum()), bad.size,
                                                          rep["bound_use"], idx))
    return rep


def assert_close(got, ref, what=""):
    """Element-wise |got - ref| <= ATOL + RTOL * |ref| (the decode tolerance)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError("%s: %d of %d elements out of tolerance (max abs err %.3g); first %s"
                             % (what, int(bad.sum()), bad.size, float(err.max()), idx))
    return float(err.max())


def check_parity(out, wl, expected, spread, what, flags=0, rows=None, allclose=True):
    """The decode tolerance (|g - o| <= 4e-3 + 1e-2 |o|) and the rounding
    bound of rounding_report on the same elements; rows selects the output
    rows the oracle was evaluated on.  Returns the rounding figures."""
    bits = bits_of(out)
    if rows is not None:
        bits = bits[rows]
    if allclose:
        assert_close(bits_to_f64(bits, wl.dtype), expected, what)
    return rounding_report(bits, expected, spread, wl.dtype, weight_roundoff(wl, flags), what)
