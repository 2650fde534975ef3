"""Seeded synthetic workloads for paged decode attention.

Input generation only: the shared source of inputs for both the CUDA library
and the fp64 oracle.  It builds block tables (through the block bookkeeping in
``workloads.blocks``), sequence lengths, query vectors, pool contents and the
step's new K/V rows.  It holds none of the method's arithmetic: no flat slot
numbers, no attention, no cache writes.

Shapes follow the layer shapes the pages name (Llama-2-7B, Llama-3-8B and
Qwen2-0.5B in "vLLM self-hosted", section "How big the KV cache is"; a
70B-class layer with 8 KV heads), blocks of 16 tokens ("vLLM Framework and
Inference Engine Design", "vLLM anatomy", "vLLM"), and ragged lengths.

Conventions:
* pools are uint16 bit patterns [num_blocks, block_size, num_kv_heads, head_dim]
  holding binary16 (F16) or bfloat16 (BF16) values, or, for an FP8 KV cache,
  uint8 E4M3 codes of the same shape with one scale for K and one for V;
* ``seq_lens`` count the tokens after the step's cache write: the step writes
  the K/V of position seq_lens[i] - 1 (and, for the shared-prefix workload, of
  the whole divergent suffix) and then decodes the query of the newest token;
* block-table entries past ceil(seq_len / block_size) are -1.
"""
import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from .blocks import BlockPool, Sequence

F16 = 0
BF16 = 1
FP8 = 2   # E4M3 KV cache (the pools only; q and the new K/V rows stay 16-bit)
DTYPE_NAMES = {F16: "f16", BF16: "bf16", FP8: "e4m3"}


# ---------------------------------------------------------------------------
# float32 -> 16-bit storage patterns (round to nearest even)
# ---------------------------------------------------------------------------

def to_bits(x, dtype):
    """Finite float32 values -> binary16 / bfloat16 bit patterns, round to
    nearest even (binary16 through numpy's own conversion)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    u = x.view(np.uint32)
    return ((u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))))
            >> np.uint32(16)).astype(np.uint16)


NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}


def _normal_bits_into(out, sigma, dtype, seed, rows=None, chunk_rows=256, threads=8):
    """Fill rows of ``out`` (uint16; the first axis indexes rows) with
    N(0, sigma^2) patterns.  ``rows`` lists the row indices to fill, in
    generation order (default: all rows in order).

    Each chunk of rows has its own generator spawned from ``seed``, so the
    values do not depend on the number of threads."""
    if rows is None:
        rows = np.arange(out.shape[0])
    n = len(rows)
    n_chunks = max(1, -(-n // chunk_rows))
    if not isinstance(seed, np.random.SeedSequence):
        seed = np.random.SeedSequence(seed)
    children = seed.spawn(n_chunks)
    inner = out.shape[1:]

    def work(c):
        lo, hi = c * chunk_rows, min(n, (c + 1) * chunk_rows)
        g = np.random.default_rng(children[c])
        v = np.empty((hi - lo,) + inner, np.float32)
        g.standard_normal(out=v, dtype=np.float32)
        if sigma != 1.0:
            v *= np.float32(sigma)
        out[rows[lo:hi]] = to_bits(v, dtype)

    if n_chunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(n_chunks)))


def random_e4m3_codes(rng, shape, exp_mean=12.5, exp_sd=1.2):
    """Random E4M3 codes (no NaN codes) built bit field by bit field: a
    random sign, an exponent field drawn around exp_mean (12.5: magnitudes
    near 2^5.5, the bulk of a tensor quantized with scale amax / 448) and a
    uniform 3-bit fraction."""
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, n, dtype=np.uint8) << np.uint8(7)
    e = np.clip(np.rint(rng.normal(exp_mean, exp_sd, n)), 0, 15).astype(np.uint8)
    f = rng.integers(0, 8, n, dtype=np.uint8)
    f[(e == 15) & (f == 7)] = 6   # S.1111.111 is NaN
    return (sign | (e << np.uint8(3)) | f).reshape(shape)


def _e4m3_codes_into(out, seed, rows, chunk_rows=256, threads=8):
    """Fill rows of a uint8 pool with random_e4m3_codes, one generator per
    chunk of rows spawned from ``seed``."""
    n = len(rows)
    n_chunks = max(1, -(-n // chunk_rows))
    if not isinstance(seed, np.random.SeedSequence):
        seed = np.random.SeedSequence(seed)
    children = seed.spawn(n_chunks)
    inner = out.shape[1:]

    def work(c):
        lo, hi = c * chunk_rows, min(n, (c + 1) * chunk_rows)
        out[rows[lo:hi]] = random_e4m3_codes(np.random.default_rng(children[c]),
                                             (hi - lo,) + inner)

    if n_chunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(n_chunks)))


E4M3_NAN = 0x7F


@dataclass
class Workload:
    name: str
    dtype: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray          # int32 [N], after the step's writes
    block_tables: np.ndarray      # int32 [N, stride]
    q: np.ndarray                 # uint16 [N, Hq, D]
    k_cache: np.ndarray           # uint16 [nb, B, H_kv, D], before the step
    v_cache: np.ndarray
    new_seq: np.ndarray           # int32 [n_new]: sequence of each new token
    new_pos: np.ndarray           # int32 [n_new]: its position in the sequence
    k_new: np.ndarray             # uint16 [n_new, H_kv, D]
    v_new: np.ndarray
    copy_pairs: np.ndarray        # int32 [n_pairs, 2] (src, dst), applied before the write
    seed: int
    recipe: str
    shared_blocks: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    kv_dtype: int = -1            # FP8 for an E4M3 pool; -1: the pools hold `dtype`
    window: int = 0               # sliding-window attention over the last `window` tokens (0: none)
    # multi-query steps (chunked prefill): q holds every new token's rows
    # [total_q, Hq, D]; sequence i's are rows [query_start[i], query_start[i+1])
    query_start: np.ndarray = None
    k_scale: float = 1.0          # E4M3 pools: value = e4m3(code) * scale
    v_scale: float = 1.0

    @property
    def fp8(self):
        return self.kv_dtype == FP8

    @property
    def num_seqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_seq_len(self):
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def scale(self):
        # 1/sqrt(head_dim), as an fp32 value
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))

    @property
    def elem_bytes(self):
        return 1 if self.fp8 else 2


def _tables_from_lengths(lens, B, pool, window=0):
    seqs = []
    for T in lens:
        s = Sequence(pool, B)
        s.reserve(int(T))
        if window > 0:
            s.release_before_window(window)
        seqs.append(s)
    stride = max([len(s.table) for s in seqs] + [1])
    bt = np.full((len(seqs), stride), -1, np.int32)
    for i, s in enumerate(seqs):
        bt[i, :len(s.table)] = s.table
    return bt


def _garbage_fill(k_cache, v_cache, valid_mask, dtype):
    nan = E4M3_NAN if k_cache.dtype == np.uint8 else NAN_BITS[dtype]
    k_cache[~valid_mask] = nan
    v_cache[~valid_mask] = nan


def valid_slot_mask(wl):
    """[num_blocks, B] True where a slot holds a token the step's decode reads."""
    B = wl.block_size
    mask = np.zeros((wl.num_blocks, B), bool)
    for i, T in enumerate(wl.seq_lens):
        T = int(T)
        s0 = max(0, T - wl.window) if wl.window > 0 else 0
        nblk = -(-T // B)
        for j in range(s0 // B, nblk):
            p = wl.block_tables[i, j]
            lo = max(0, s0 - j * B)
            n = min(B, T - j * B)
            mask[p, lo:n] = True
    return mask


def decode_workload(name, dtype, Hq, H_kv, D, B, num_blocks, lens, seed, q_sigma=1.0,
                    kv_sigma=1.0, garbage="random", recipe="", fp8_scales=None, window=0):
    """One new token per sequence at position T_i - 1, then decode.

    Blocks are popped, sequence by sequence and block by block, from a free
    list in the order of a seeded permutation of the pool.  With
    fp8_scales = (k_scale, v_scale) the pools hold random E4M3 codes."""
    lens = np.asarray(lens, dtype=np.int32)
    ss = np.random.SeedSequence(seed)
    s_perm, s_q, s_k, s_v, s_nk, s_nv = ss.spawn(6)
    free_order = np.random.default_rng(s_perm).permutation(num_blocks)
    pool = BlockPool(num_blocks, free_order)
    bt = _tables_from_lengths(lens, B, pool, window)
    N = lens.shape[0]
    q = np.empty((N, Hq, D), np.uint16)
    _normal_bits_into(q, q_sigma, dtype, s_q)
    used = bt[bt >= 0]
    if fp8_scales is None:
        k_cache = np.zeros((num_blocks, B, H_kv, D), np.uint16)
        v_cache = np.zeros((num_blocks, B, H_kv, D), np.uint16)
        # values of the allocated blocks, in allocation order
        _normal_bits_into(k_cache, kv_sigma, dtype, s_k, rows=used)
        _normal_bits_into(v_cache, kv_sigma, dtype, s_v, rows=used)
    else:
        k_cache = np.zeros((num_blocks, B, H_kv, D), np.uint8)
        v_cache = np.zeros((num_blocks, B, H_kv, D), np.uint8)
        _e4m3_codes_into(k_cache, s_k, used)
        _e4m3_codes_into(v_cache, s_v, used)
    new_seq = np.arange(N, dtype=np.int32)
    new_pos = (lens - 1).astype(np.int32)
    k_new = np.empty((N, H_kv, D), np.uint16)
    v_new = np.empty((N, H_kv, D), np.uint16)
    _normal_bits_into(k_new, kv_sigma, dtype, s_nk)
    _normal_bits_into(v_new, kv_sigma, dtype, s_nv)
    wl = Workload(name, dtype, Hq, H_kv, D, B, num_blocks, lens, bt, q, k_cache, v_cache,
                  new_seq, new_pos, k_new, v_new, np.zeros((0, 2), np.int32), seed, recipe)
    wl.window = int(window)
    if fp8_scales is not None:
        wl.kv_dtype = FP8
        wl.k_scale = float(np.float32(fp8_scales[0]))
        wl.v_scale = float(np.float32(fp8_scales[1]))
    if garbage == "nan":
        _garbage_fill(k_cache, v_cache, valid_slot_mask(wl), dtype)
    return wl


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def tiny(seed=1, garbage="random"):
    """4 sequences of lengths [7, 8, 9, 33] (after the write), 8 query heads =
    8 KV heads, head_dim 64, block size 4, fp16, a pool of 32 blocks."""
    return decode_workload("tiny", F16, 8, 8, 64, 4, 32, [7, 8, 9, 33], seed,
                           garbage=garbage,
                           recipe="q,k,v ~ N(0,1) fp16; blocks from a seeded permutation of 32")


def llama2_7b(seed=2, num_seqs=64, garbage="random"):
    """Llama-2-7B layer: 32 q heads = 32 KV heads, head_dim 128, fp16, block
    16; lengths uniform in [1, 2048]; a pool of 10,000 blocks."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 101]))
    lens = rng.integers(1, 2048, size=num_seqs, endpoint=True)
    return decode_workload("llama2-7b", F16, 32, 32, 128, 16, 10_000, lens, seed,
                           garbage=garbage,
                           recipe="T ~ U[1,2048]; q,k,v ~ N(0,1) fp16; free list = seeded "
                                  "permutation of 10,000 blocks")


LOGNORMAL_SIGMA = 0.632
LOGNORMAL_MU = math.log(400.0) - LOGNORMAL_SIGMA ** 2 / 2


def llama3_8b_lengths(seed=3, num_seqs=256):
    rng = np.random.default_rng(np.random.SeedSequence([seed, 103]))
    lens = np.rint(rng.lognormal(LOGNORMAL_MU, LOGNORMAL_SIGMA, size=num_seqs))
    return np.clip(lens, 16, 4096).astype(np.int32)


def llama3_8b(seed=3, num_seqs=256, garbage="random", num_blocks=40_000):
    """Llama-3-8B GQA layer: 32 q heads / 8 KV heads, head_dim 128, bf16, block
    16; 256 sequences with lognormal lengths (mean about 400, sigma 0.632 in
    log space), clipped to [16, 4096]; 40,000-block pool; K/V ~ N(0, 0.5^2)."""
    lens = llama3_8b_lengths(seed, num_seqs)
    return decode_workload("llama3-8b-gqa", BF16, 32, 8, 128, 16, num_blocks, lens, seed,
                           q_sigma=1.0, kv_sigma=0.5, garbage=garbage,
                           recipe="T ~ round(lognormal(ln400 - 0.632^2/2, 0.632)) clipped to "
                                  "[16,4096]; q ~ N(0,1), k,v ~ N(0,0.25) bf16; free list = "
                                  "seeded permutation of 40,000 blocks")


# E4M3 scales of the FP8 workloads: K/V ~ N(0, 0.5^2) quantized with
# scale amax / 448 would put sigma near 2^6 codes' magnitude; 2^-7 does that.
FP8_SCALES = (2.0 ** -7, 2.0 ** -7)


def llama3_8b_fp8(seed=3, num_seqs=256, garbage="random", num_blocks=40_000):
    """The Llama-3-8B GQA layer with an FP8 (E4M3) KV cache: same lengths,
    tables and queries as llama3-8b-gqa; random E4M3 codes in the pool,
    k_scale = v_scale = 2^-7; the step's new K/V rows are bf16 and are
    quantized by the write."""
    lens = llama3_8b_lengths(seed, num_seqs)
    return decode_workload("llama3-8b-gqa-fp8", BF16, 32, 8, 128, 16, num_blocks, lens, seed,
                           q_sigma=1.0, kv_sigma=0.5, garbage=garbage, fp8_scales=FP8_SCALES,
                           recipe="llama3-8b-gqa lengths and tables; pool = random E4M3 "
                                  "codes (sign uniform, exponent field ~ round(N(12.5, "
                                  "1.2)), fraction uniform); k_scale = v_scale = 2^-7")


def mistral_7b_swa(seed=6, num_seqs=64, lo=4_096, hi=16_384, window=4_096, garbage="random",
                   num_blocks=20_000):
    """Sliding-window layer of Mistral 7B v0.1 (the model and its 4,096-token
    window are the pages' example, "How does it support prompts of arbitrary
    length? Does it have a sliding window?"; its layer shape, 32 q heads / 8
    KV heads / head_dim 128, is the public model card's): bf16, 16-token
    blocks, lengths uniform in [4,096, 16,384]; every sequence keeps only the
    blocks that reach into its window, the others are released back to the
    pool (table entries -1), so at most ceil(W/B) + 1 = 257 blocks a sequence."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 106]))
    lens = rng.integers(lo, hi + 1, size=num_seqs).astype(np.int32)
    return decode_workload("mistral-7b-swa", BF16, 32, 8, 128, 16, num_blocks, lens, seed,
                           q_sigma=1.0, kv_sigma=0.5, garbage=garbage, window=window,
                           recipe="T ~ U[4096, 16384]; window 4096; blocks before the window "
                                  "released to the free list (table entries -1); q ~ N(0,1), "
                                  "k,v ~ N(0,0.25) bf16; free list = seeded permutation of "
                                  "20,000 blocks")


def long_context_70b(seed=5, num_seqs=32, lo=16_384, hi=32_768, garbage="random"):
    """70B-class long-context layer: 64 q heads / 8 KV heads, head_dim 128,
    bf16, block 16; lengths uniform in [16,384, 32,768]; the pool has 10%
    free blocks interleaved at random (pool = ceil(needed / 0.9))."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 105]))
    lens = rng.integers(lo, hi, size=num_seqs, endpoint=True).astype(np.int32)
    needed = int(sum(-(-int(T) // 16) for T in lens))
    num_blocks = -(-needed * 10 // 9)
    return decode_workload("70b-long-context", BF16, 64, 8, 128, 16, num_blocks, lens, seed,
                           garbage=garbage,
                           recipe="T ~ U[16384,32768]; q,k,v ~ N(0,1) bf16; pool = "
                                  "ceil(needed/0.9) blocks, free list = seeded permutation")


def shared_prefix(seed=4, num_seqs=12, prefix=1800, suffix_hi=300, num_blocks=1024,
                  garbage="random"):
    """Qwen2-0.5B shape (14 q heads / 2 KV heads, head_dim 64, fp16, block 16):
    num_seqs sequences share the blocks of one prefix; each then writes its own
    suffix of U[1, suffix_hi] tokens.  The first write of each sharer into the
    partially filled last shared block triggers a copy-on-write; the last
    writer finds a reference count of 1 and writes in place."""
    dtype, Hq, H_kv, D, B = F16, 14, 2, 64, 16
    ss = np.random.SeedSequence(seed)
    s_perm, s_len, s_q, s_k, s_v, s_nk, s_nv = ss.spawn(7)
    free_order = np.random.default_rng(s_perm).permutation(num_blocks)
    pool = BlockPool(num_blocks, free_order)
    root = Sequence(pool, B)
    root.reserve(prefix)
    shared = list(root.table)
    seqs = [root] + [root.fork() for _ in range(num_seqs - 1)]
    suffix = np.random.default_rng(s_len).integers(1, suffix_hi, size=num_seqs, endpoint=True)
    pairs = []
    for s, n in zip(seqs, suffix):
        pairs += s.reserve(int(n))
    lens = np.array([s.num_tokens for s in seqs], np.int32)
    stride = max(len(s.table) for s in seqs)
    bt = np.full((num_seqs, stride), -1, np.int32)
    for i, s in enumerate(seqs):
        bt[i, :len(s.table)] = s.table
    q = np.empty((num_seqs, Hq, D), np.uint16)
    _normal_bits_into(q, 1.0, dtype, s_q)
    k_cache = np.zeros((num_blocks, B, H_kv, D), np.uint16)
    v_cache = np.zeros((num_blocks, B, H_kv, D), np.uint16)
    # every block in use gets values before the step; the prefix blocks hold
    # the shared context, the others hold stale contents the step overwrites
    used = np.unique(bt[bt >= 0])
    _normal_bits_into(k_cache, 1.0, dtype, s_k, rows=used)
    _normal_bits_into(v_cache, 1.0, dtype, s_v, rows=used)
    new_seq = np.concatenate([np.full(int(n), i, np.int32) for i, n in enumerate(suffix)])
    new_pos = np.concatenate([np.arange(prefix, prefix + int(n), dtype=np.int32)
                              for n in suffix])
    k_new = np.empty((new_seq.size, H_kv, D), np.uint16)
    v_new = np.empty((new_seq.size, H_kv, D), np.uint16)
    _normal_bits_into(k_new, 1.0, dtype, s_nk)
    _normal_bits_into(v_new, 1.0, dtype, s_nv)
    wl = Workload("qwen2-0.5b-shared-prefix", dtype, Hq, H_kv, D, B, num_blocks, lens, bt, q,
                  k_cache, v_cache, new_seq, new_pos, k_new, v_new,
                  np.array(pairs, np.int32).reshape(-1, 2), seed,
                  "12 sequences share a 1,800-token prefix (113 blocks, the last holding 8 "
                  "tokens); suffix ~ U[1,300]; q,k,v ~ N(0,1) fp16; 1,024-block pool",
                  shared_blocks=np.array(shared, np.int32))
    if garbage == "nan":
        # only slots nobody reads after the step get NaN; the suffix slots are
        # written by the step itself
        mask = valid_slot_mask(wl)
        k_cache[~mask] = NAN_BITS[dtype]
        v_cache[~mask] = NAN_BITS[dtype]
    return wl


def prefill_workload(name, dtype, Hq, H_kv, D, B, num_blocks, prefix_lens, chunk_lens, seed,
                     q_sigma=1.0, kv_sigma=1.0, garbage="random", recipe=""):
    """A chunked-prefill step ("vLLM Framework and Inference Engine Design",
    "How does it support prompts of arbitrary length?": a long prompt is
    processed in chunks, with other requests' decode tokens in the same batch):
    sequence i holds prefix_lens[i] cached tokens and brings chunk_lens[i] >= 1
    new tokens (1 = a decode token).  The step writes the new tokens' K/V at
    positions prefix_lens[i] .. prefix_lens[i] + chunk_lens[i] - 1, then every
    new token's query attends causally through the block table."""
    prefix_lens = np.asarray(prefix_lens, np.int32)
    chunk_lens = np.asarray(chunk_lens, np.int32)
    assert np.all(chunk_lens >= 1) and np.all(prefix_lens >= 0)
    lens = prefix_lens + chunk_lens
    ss = np.random.SeedSequence(seed)
    s_perm, s_q, s_k, s_v, s_nk, s_nv = ss.spawn(6)
    free_order = np.random.default_rng(s_perm).permutation(num_blocks)
    pool = BlockPool(num_blocks, free_order)
    bt = _tables_from_lengths(lens, B, pool)
    total = int(chunk_lens.sum())
    q = np.empty((total, Hq, D), np.uint16)
    _normal_bits_into(q, q_sigma, dtype, s_q)
    k_cache = np.zeros((num_blocks, B, H_kv, D), np.uint16)
    v_cache = np.zeros((num_blocks, B, H_kv, D), np.uint16)
    used = bt[bt >= 0]
    _normal_bits_into(k_cache, kv_sigma, dtype, s_k, rows=used)
    _normal_bits_into(v_cache, kv_sigma, dtype, s_v, rows=used)
    new_seq = np.repeat(np.arange(lens.size, dtype=np.int32), chunk_lens)
    new_pos = np.concatenate([np.arange(p, p + c, dtype=np.int32)
                              for p, c in zip(prefix_lens, chunk_lens)])
    k_new = np.empty((total, H_kv, D), np.uint16)
    v_new = np.empty((total, H_kv, D), np.uint16)
    _normal_bits_into(k_new, kv_sigma, dtype, s_nk)
    _normal_bits_into(v_new, kv_sigma, dtype, s_nv)
    wl = Workload(name, dtype, Hq, H_kv, D, B, num_blocks, lens, bt, q, k_cache, v_cache,
                  new_seq, new_pos, k_new, v_new, np.zeros((0, 2), np.int32), seed, recipe)
    wl.query_start = np.concatenate([[0], np.cumsum(chunk_lens)]).astype(np.int32)
    if garbage == "nan":
        _garbage_fill(k_cache, v_cache, valid_slot_mask(wl), dtype)
    return wl


def random_prefill(seed, dtype, Hq, H_kv, D, B, prefix_lens, chunk_lens, spare_blocks=7,
                   garbage="random", q_sigma=1.0, kv_sigma=1.0):
    """A chunked-prefill parity case of any shape."""
    lens = np.asarray(prefix_lens) + np.asarray(chunk_lens)
    need = int(sum(-(-int(T) // B) for T in lens))
    return prefill_workload("random-prefill", dtype, Hq, H_kv, D, B, need + spare_blocks,
                            prefix_lens, chunk_lens, seed, q_sigma=q_sigma, kv_sigma=kv_sigma,
                            garbage=garbage, recipe="parity case")


def llama3_8b_chunked_prefill(seed=7, num_seqs=16, chunk=512, garbage="random",
                              num_blocks=8_000):
    """Llama-3-8B GQA layer (32 q / 8 KV heads, head_dim 128, bf16, block 16),
    a chunked-prefill step: 16 prompts each bring a 512-token chunk (an 8,192-
    token step budget) on top of lognormal cached prefixes (median about 1,300
    tokens, clipped to [0, 6,144]) -- a long prompt's later chunks or a
    prefix-cache hit."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 107]))
    prefix = np.clip(np.rint(rng.lognormal(np.log(1300), 0.8, size=num_seqs)), 0,
                     6144).astype(np.int32)
    chunks = np.full(num_seqs, chunk, np.int32)
    return prefill_workload("llama3-8b-chunked-prefill", BF16, 32, 8, 128, 16, num_blocks,
                            prefix, chunks, seed, kv_sigma=0.5, garbage=garbage,
                            recipe="16 sequences x 512-token chunks on lognormal(ln 1300, 0.8) "
                                   "prefixes clipped to [0, 6144]; q ~ N(0,1), k,v ~ N(0,0.25) "
                                   "bf16; 8,000-block pool")


def random_workload(seed, dtype, Hq, H_kv, D, B, lens, num_blocks=None, q_sigma=1.0,
                    kv_sigma=1.0, garbage="random", spare_blocks=7, fp8_scales=None, window=0):
    """A parity-test case of any shape: blocks scattered through a pool with
    spare_blocks extra blocks.  With a window, blocks wholly before it are
    released (table entries -1) once each sequence is built."""
    lens = np.asarray(lens, np.int32)
    need = int(sum(-(-int(T) // B) for T in lens))
    if num_blocks is None:
        num_blocks = need + spare_blocks
    return decode_workload("random", dtype, Hq, H_kv, D, B, num_blocks, lens, seed,
                           q_sigma=q_sigma, kv_sigma=kv_sigma, garbage=garbage,
                           recipe="parity case", fp8_scales=fp8_scales, window=window)


CONFIGS = {
    "tiny": tiny,
    "llama2-7b": llama2_7b,
    "llama3-8b-gqa": llama3_8b,
    "qwen2-0.5b-shared-prefix": shared_prefix,
    "70b-long-context": long_context_70b,
    "llama3-8b-gqa-fp8": llama3_8b_fp8,
    "mistral-7b-swa": mistral_7b_swa,
    "llama3-8b-chunked-prefill": llama3_8b_chunked_prefill,
}
