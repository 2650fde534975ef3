"""Benchmark of the paged decode step on GB300.

A step is one pass of the hot path over one batch: copy-on-write block copies
(shared-prefix workload only), slot mapping, cache write of the step's new
K/V, and paged decode attention (one kernel; split contexts merged in-grid).  The
default workload is the Llama-3-8B GQA decode layer (256 sequences, lognormal
lengths with mean about 400, 32 q heads / 8 KV heads, head_dim 128, bf16,
16-token blocks, 40,000-block pool).

Prints ONE JSON line (rank 0).  `value` is sequence-steps per second over all
ranks; `roofline` reports the decode kernels' achieved HBM bandwidth
(algorithmic bytes / CUDA-event time) against the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "Paged decode attention: achieved HBM GB/s vs GB300 peak; seq-steps/sec"
UNIT = "seq-steps/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DATASHEET_HBM_GBS = 7900.0   # nominal GB300 HBM3e figure, for context only
L2_FLUSH_BYTES = 512 << 20
CLOCK_SOAK_S = 0.5   # untimed replays of the step under the clock sampler before timing
KERNEL_SOURCES = ["pa_decode_kernel.cuh", "pa_decode_fp8.cuh", "pa_device.cuh",
                  "pa_decode_variants.cuh", "pa_decode.cu"]
PREFILL_SOURCES = ["pa_prefill.cu", "pa_device.cuh"]


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def algorithmic_bytes(wl):
    """Bytes the step must move, per the method (no implementation overhead).

    decode: every used K and V row of every KV head (2 * e * H_kv * D * sum T),
    the queries and outputs (2 * N * Hq * D * e), one block-table entry per
    used block and one length per sequence.  cache write: read the new K/V and
    write them, plus one int64 slot per token (and the two int32 inputs of the
    slot mapping).  copy-on-write: read and write each copied block, K and V.
    KV elements take wl.elem_bytes (1 for an E4M3 cache); queries, outputs and
    the new K/V rows are 16-bit."""
    e = wl.elem_bytes
    T = wl.seq_lens.astype(np.int64)
    N = wl.num_seqs
    # a sliding window attends to the last `window` tokens only
    s0 = np.maximum(T - wl.window, 0) if wl.window > 0 else np.zeros_like(T)
    kv = 2 * e * wl.num_kv_heads * wl.head_dim * int((T - s0).sum())
    qo = 2 * N * wl.num_q_heads * wl.head_dim * 2
    B = wl.block_size
    tables = 4 * int(sum(-(-int(t) // B) - int(s) // B for t, s in zip(T, s0)))
    lens = 4 * N
    if wl.query_start is not None:
        qo = 2 * int(wl.query_start[-1]) * wl.num_q_heads * wl.head_dim * 2
    decode = kv + qo + tables + lens
    n_new = wl.new_seq.size
    write = 2 * (2 + e) * n_new * wl.num_kv_heads * wl.head_dim + 8 * n_new + 16 * n_new
    cow = 2 * 2 * wl.copy_pairs.shape[0] * wl.block_size * wl.num_kv_heads * wl.head_dim * e
    return {"decode": decode, "kv": kv, "write": write, "cow": cow, "step": decode + write + cow}


def prefill_flops(wl):
    """Tensor-core work of a multi-query step, causal: every new token at
    position p scores and weights p + 1 keys, 2 D flops each for Q.K^T and
    for P.V, over all query heads."""
    qs = wl.query_start
    keys = 0
    for i, T in enumerate(wl.seq_lens.astype(np.int64)):
        L = int(qs[i + 1] - qs[i])
        first = int(T) - L + 1   # keys seen by the first new token
        keys += L * first + L * (L - 1) // 2
    return 4 * wl.head_dim * wl.num_q_heads * keys


def measured_peaks(key="hbm_gbs"):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    return (FALLBACK_HBM_GBS if key == "hbm_gbs" else FALLBACK_BF16_TFLOPS), "fallback"


def kernel_sha(sources=KERNEL_SOURCES):
    """Short hash of the sources of the kernel a traffic record was taken on."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "paged_kv_cache_72_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, prefill=False):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(workload)
    sources = PREFILL_SOURCES if prefill else KERNEL_SOURCES
    if not rec or rec.get("kernel_sha") != kernel_sha(sources):
        return None
    return rec.get("dram_bytes_per_launch")


def l2_flush(buf, k):
    """Evict the step's data from L2: write a buffer four times the L2 size,
    then read it back, so that the next step starts with a cold L2 that holds
    no dirty lines (their write-back would otherwise land in the timed step)."""
    buf.fill_(float(k % 7 + 1))
    buf.amax()


class ClockSampler:
    """nvidia-smi samples (every 20 ms, read-only queries) of SM clock and
    throttle reasons, each stamped with the host time it arrived."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0:
                time.sleep(0.02)
            self.lines = []
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, region=None):
        """Summary of the samples; region = (t0, t1) host times of the timed
        region, whose samples are counted separately."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons, in_region = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            if region and region[0] <= t <= region[1]:
                in_region.append(sm[-1])
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "samples_in_timed_region": len(in_region),
                "sm_mhz_in_timed_region": statistics.median(in_region) if in_region else None,
                "reasons": sorted(reasons),
                "window": "every 20 ms over an untimed soak of the same step (about %.1f s, "
                          "graph replays with the L2 flush) running straight into the timed "
                          "region, and the timed region itself" % CLOCK_SOAK_S}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

class Step:
    """Device-resident inputs and the step as calls into the C ABI."""

    def __init__(self, wl, device):
        import torch
        import paged_kv_cache_72_gb300 as pa
        self.pa, self.torch, self.wl = pa, torch, wl
        td = torch.float16 if wl.dtype == W.F16 else torch.bfloat16

        def up(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(td)

        if wl.fp8:   # uint8 E4M3 codes
            self.k_cache = torch.from_numpy(wl.k_cache).to(device)
            self.v_cache = torch.from_numpy(wl.v_cache).to(device)
        else:
            self.k_cache = up(wl.k_cache)
            self.v_cache = up(wl.v_cache)
        self.q = up(wl.q)
        self.k_new = up(wl.k_new)
        self.v_new = up(wl.v_new)
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        self.new_seq = torch.from_numpy(wl.new_seq).to(device)
        self.new_pos = torch.from_numpy(wl.new_pos).to(device)
        self.pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, np.int32)).to(device)
        self.slots = torch.empty(wl.new_seq.size, dtype=torch.int64, device=device)
        self.out = torch.empty_like(self.q)
        nbytes = pa.pa_decode_workspace_size(wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                             wl.block_size, W.FP8 if wl.fp8 else wl.dtype)
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        # a step's lengths and block tables are in place before its first
        # kernel, so the decode may read them while the cache write drains
        self.flags = pa.PA_DECODE_TABLES_READY
        self.query_start = (None if wl.query_start is None
                            else torch.from_numpy(wl.query_start).to(device))
        self.pf_ws = torch.zeros(256, dtype=torch.uint8, device=device)
        self.ev0 = torch.cuda.Event(enable_timing=True)
        self.ev1 = torch.cuda.Event(enable_timing=True)
        self.decode_ms = []

    def launches_per_step(self):
        # copy-on-write (if any), the slot-mapped cache write, decode (split
        # contexts are merged inside the decode grid)
        return (1 if self.pairs.numel() else 0) + 1 + 1

    def write_phase(self):
        pa, wl = self.pa, self.wl
        if self.pairs.numel():
            pa.pa_copy_blocks(self.pairs, self.k_cache, self.v_cache, err=self.err)
        # slot mapping and cache write in one launch
        if wl.fp8:
            pa.pa_cache_write_fp8_mapped(self.k_new, self.v_new, self.block_tables, self.new_seq,
                                         self.new_pos, self.k_cache, self.v_cache, wl.k_scale,
                                         wl.v_scale, slot_mapping=self.slots, err=self.err)
        else:
            pa.pa_cache_write_mapped(self.k_new, self.v_new, self.block_tables, self.new_seq,
                                     self.new_pos, self.k_cache, self.v_cache,
                                     slot_mapping=self.slots, err=self.err)

    def decode_phase(self):
        wl = self.wl
        if wl.query_start is not None:
            self.pa.pa_prefill(self.q, self.k_cache, self.v_cache, self.block_tables,
                               self.seq_lens, self.query_start, wl.scale, out=self.out,
                               workspace=self.pf_ws, err=self.err)
        elif wl.window > 0:
            self.pa.pa_decode_window(self.q, self.k_cache, self.v_cache, self.block_tables,
                                     self.seq_lens, wl.scale, wl.window, out=self.out,
                                     workspace=self.workspace, flags=self.flags, err=self.err)
        elif wl.fp8:
            self.pa.pa_decode_fp8(self.q, self.k_cache, self.v_cache, self.block_tables,
                                  self.seq_lens, wl.scale, wl.k_scale, wl.v_scale, out=self.out,
                                  workspace=self.workspace, flags=self.flags, err=self.err)
        else:
            self.pa.pa_decode(self.q, self.k_cache, self.v_cache, self.block_tables,
                              self.seq_lens, wl.scale, out=self.out, workspace=self.workspace,
                              flags=self.flags, err=self.err)

    def run(self):
        self.write_phase()
        self.decode_phase()

    def capture(self):
        """CUDA graphs of the step and of its decode phase alone (the calls are
        the same C-ABI calls; a graph removes the per-call host cost from the
        GPU timeline, and inside the step graph each kernel may start while
        its predecessor drains)."""
        torch = self.torch
        self.g_step = torch.cuda.CUDAGraph()
        self.g_decode = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.g_step, stream=s):
                self.write_phase()
                self.decode_phase()
            with torch.cuda.graph(self.g_decode, stream=s):
                self.decode_phase()
        torch.cuda.current_stream().wait_stream(s)


def run_gpu(args, rank, world, local_rank):
    import torch
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    import paged_kv_cache_72_gb300 as pa
    kw = {"num_blocks": args.pool_blocks} if args.pool_blocks else {}
    wl = W.CONFIGS[args.workload](seed=_seed(args) + rank, **kw)
    st = Step(wl, device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    nbytes = algorithmic_bytes(wl)

    for k in range(args.warmup):
        l2_flush(flush, k)
        st.run()
    torch.cuda.synchronize()
    flags = pa.pa_get_error(st.err)
    if flags:
        raise RuntimeError("kernel reported error bits 0x%x" % flags)
    st.capture()
    for _ in range(args.warmup):
        st.g_step.replay()
        st.g_decode.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    clocks.start()
    # keep the GPU under the step's load while the sampler collects samples
    # (a timed region of a few steps lasts milliseconds, shorter than the
    # sampling period)
    t_soak = time.perf_counter()
    k = 0
    while time.perf_counter() - t_soak < CLOCK_SOAK_S:
        l2_flush(flush, k)
        st.g_step.replay()
        k += 1
        if k % 64 == 0:
            torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    t_region0 = time.perf_counter()
    # timed region: K steps (one graph each), then K decode phases alone for
    # the decode kernels' own duration; L2 flushed before each, untimed
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for k in range(args.steps):
        l2_flush(flush, k)
        ev[k][0].record()
        st.g_step.replay()
        ev[k][1].record()
    for k in range(args.steps):
        l2_flush(flush, k)
        ev[k][2].record()
        st.g_decode.replay()
        ev[k][3].record()
    torch.cuda.synchronize()
    t_region1 = time.perf_counter()
    _barrier(world)
    clk = clocks.stop(region=(t_region0, t_region1))
    flags = pa.pa_get_error(st.err)
    if flags:
        raise RuntimeError("kernel reported error bits 0x%x" % flags)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    decode_ms = [e[2].elapsed_time(e[3]) for e in ev]

    ms = statistics.mean(step_ms)
    dms = statistics.mean(decode_ms)
    ms_max = _max_over_ranks(ms, world, device)

    # end to end through the public API with host buffers: per step the
    # inputs go host -> device from pinned memory, the C-ABI calls run eagerly
    # and the output comes back
    host = {
        "q": st.q.cpu().pin_memory(), "k_new": st.k_new.cpu().pin_memory(),
        "v_new": st.v_new.cpu().pin_memory(), "block_tables": st.block_tables.cpu().pin_memory(),
        "seq_lens": st.seq_lens.cpu().pin_memory(), "new_seq": st.new_seq.cpu().pin_memory(),
        "new_pos": st.new_pos.cpu().pin_memory(), "pairs": st.pairs.cpu().pin_memory(),
    }
    if st.query_start is not None:
        host["query_start"] = st.query_start.cpu().pin_memory()
    out_host = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    e2e_ms = []
    n_e2e = min(args.steps, 200)
    for i in range(args.warmup + n_e2e):
        l2_flush(flush, i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for name, t in host.items():
            getattr(st, name).copy_(t, non_blocking=True)
        st.run()
        out_host.copy_(st.out, non_blocking=True)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e = statistics.mean(e2e_ms)
    e2e_max = _max_over_ranks(e2e, world, device)

    peak, peak_kind = measured_peaks()
    achieved = nbytes["decode"] / (dms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload, prefill=wl.query_start is not None)
    if wl.query_start is not None:
        # a dense contraction: its roofline is the tensor rate (the kernel
        # timed alone: the burst figure)
        flops = prefill_flops(wl)
        tpeak, tkind = measured_peaks("bf16_tflops")
        tach = flops / (dms * 1e-3) / 1e12
        roof = {
            "bound": "tensor", "achieved": round(tach, 1), "peak": tpeak, "unit": "TFLOP/s",
            "frac": round(tach / tpeak, 4), "traffic": traffic,
            "peak_source": tkind + " (MEASURED_PEAKS.json bf16_tflops, cuBLAS bf16 burst)",
            "kernel": ("pa_prefill: paged_prefill_tc_kernel (tcgen05.mma, TMEM accumulators)"
                       if pa.pa_prefill_kernel(wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                               wl.block_size, wl.dtype, wl.num_seqs)
                       == pa.PA_PREFILL_TENSOR_CORE
                       else "pa_prefill: paged_prefill_kernel (warp-level mma.sync)"),
            "algorithmic_flops_per_launch": flops,
            "kv_gbs": round(achieved, 1),
        }
        return {
            "wl": wl, "ms": ms_max, "ms_local": ms, "decode_ms": dms, "e2e_ms": e2e_max,
            "h2d": h2d, "d2h": d2h, "bytes": nbytes, "clocks": clk,
            "launches": st.launches_per_step() * args.steps, "roofline": roof,
        }
    return {
        "wl": wl, "ms": ms_max, "ms_local": ms, "decode_ms": dms, "e2e_ms": e2e_max,
        "h2d": h2d, "d2h": d2h, "bytes": nbytes, "clocks": clk,
        "launches": st.launches_per_step() * args.steps,
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "kernel": "pa_decode: paged_decode_kernel",
            "algorithmic_bytes_per_launch": nbytes["decode"],
            "frac_of_datasheet_7.9TBps": round(achieved / DATASHEET_HBM_GBS, 4),
        },
    }


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world, device):
    """The slowest rank's value (each rank runs its own replica; the job's
    time is that of the slowest).  Only this timing scalar crosses ranks."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    if dist.get_backend() != "nccl":
        device = "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(num_seqs, world, ms_max):
    """Weak scaling: every rank decodes its own batch of num_seqs sequences;
    the job's throughput is all ranks' sequences over the slowest rank's step."""
    return num_seqs * world / (ms_max * 1e-3)


# --------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# --------------------------------------------------------------------------

def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleStep:
    """The fp64 oracle's step (cache write of the sampled sequences' new tokens
    + decode of all their query heads) on the host cores."""

    def __init__(self, wl, threads=0):
        import oracle
        self.oracle, self.wl = oracle, wl
        self.cores = threads if threads > 0 else cores()
        self.kc, self.vc = wl.k_cache.copy(), wl.v_cache.copy()
        self.slots = oracle.slot_mapping(wl.block_tables, wl.new_seq, wl.new_pos, wl.block_size)

    def run(self, n):
        wl, o = self.wl, self.oracle
        ids = np.arange(n, dtype=np.int32)
        mask = np.isin(wl.new_seq, ids)
        t0 = time.perf_counter()
        if wl.query_start is not None:
            # the sampled sequences' chunks: their new tokens' K/V, then their rows
            o.cache_write(self.kc, self.vc, wl.k_new[mask], wl.v_new[mask], self.slots[mask])
            qs = wl.query_start
            o.paged_prefill(wl.q[qs[0]:qs[n]], self.kc, self.vc, wl.dtype, wl.block_tables[:n],
                            wl.seq_lens[:n], qs[:n + 1], wl.scale, threads=self.cores)
        elif wl.window > 0:
            o.cache_write(self.kc, self.vc, wl.k_new[mask], wl.v_new[mask], self.slots[mask])
            o.paged_decode_window(wl.q, self.kc, self.vc, wl.dtype, wl.block_tables,
                                  wl.seq_lens, wl.window, wl.scale, seq_ids=ids,
                                  threads=self.cores)
        elif wl.fp8:
            o.cache_write_fp8(self.kc, self.vc, wl.k_new[mask], wl.v_new[mask], wl.dtype,
                              self.slots[mask], wl.k_scale, wl.v_scale)
            o.paged_decode_fp8(wl.q, self.kc, self.vc, wl.dtype, wl.k_scale, wl.v_scale,
                               wl.block_tables, wl.seq_lens, wl.scale, seq_ids=ids,
                               threads=self.cores)
        else:
            o.cache_write(self.kc, self.vc, wl.k_new[mask], wl.v_new[mask], self.slots[mask])
            o.paged_decode(wl.q, self.kc, self.vc, wl.dtype, wl.block_tables, wl.seq_lens,
                           wl.scale, seq_ids=ids, threads=self.cores)
        return time.perf_counter() - t0

    def sample_size(self, budget_s):
        """Sequences whose step fits in about budget_s seconds."""
        probe = min(self.wl.num_seqs, 4)
        per_seq = max(self.run(probe) / probe, 1e-6)
        return int(min(self.wl.num_seqs, max(1, budget_s / per_seq)))


def oracle_rate(wl, budget_s, threads=0):
    """Sequence-steps per second of the oracle over about budget_s seconds
    (threads: host threads, 0 for every core the process may use)."""
    os_ = OracleStep(wl, threads)
    n = os_.sample_size(min(budget_s, 2.0))
    done, t_total, reps = 0, 0.0, 0
    while t_total < budget_s and reps < 1000:
        t_total += os_.run(n)
        done += n
        reps += 1
    sample = "%d of %d sequences x %d repetition(s): cache write of their new tokens + fp64 " \
             "decode of all their query heads" % (n, wl.num_seqs, reps)
    return done / t_total, sample, t_total, os_.cores


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = W.CONFIGS[args.workload](seed=_seed(args))
    os_ = OracleStep(wl)
    # the whole run stays within about two minutes of CPU time
    per_step = min(args.ref_step_seconds, max(0.05, 120.0 / (args.steps + args.warmup)))
    n = os_.sample_size(per_step)
    rates = []
    for i in range(args.warmup + args.steps):
        t = os_.run(n)
        if i >= args.warmup:
            rates.append(n / t)
    value = statistics.mean(rates)
    sample = "%d of %d sequences per step: cache write of their new tokens + fp64 decode of " \
             "all their query heads" % (n, wl.num_seqs)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": _config(wl, args),
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": os_.cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


DEFAULT_SEEDS = {"tiny": 1, "llama2-7b": 2, "llama3-8b-gqa": 3, "qwen2-0.5b-shared-prefix": 4,
                 "70b-long-context": 5, "llama3-8b-gqa-fp8": 3, "mistral-7b-swa": 6,
                 "llama3-8b-chunked-prefill": 7}


def run_swap(args):
    """Block swap bandwidth: --swap-blocks blocks of the workload's pools out
    to a pinned host pool and back in, one C-ABI call each way per step; the
    link's own rate is a contiguous device -> pinned host copy of the same
    bytes on the same stream."""
    import torch
    import paged_kv_cache_72_gb300 as pa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    wl = W.CONFIGS[args.workload](seed=_seed(args))
    st = Step(wl, device)
    used = np.unique(wl.block_tables[wl.block_tables >= 0]).astype(np.int32)
    n = min(args.swap_blocks, used.size)
    hk = torch.empty((n,) + tuple(st.k_cache.shape[1:]), dtype=st.k_cache.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_pairs = torch.from_numpy(np.stack([used[:n], np.arange(n)], 1).astype(np.int32)).cuda()
    in_pairs = torch.from_numpy(np.stack([np.arange(n), used[:n]], 1).astype(np.int32)).cuda()
    nbytes = 2 * n * st.k_cache[0].numel() * st.k_cache.element_size()   # K and V, one way
    flat = st.k_cache[:2 * n].reshape(-1) if 2 * n <= st.k_cache.shape[0] else None
    link_host = torch.empty(nbytes // st.k_cache.element_size(),
                            dtype=st.k_cache.dtype).pin_memory()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    t_out, t_in, t_link = [], [], []
    for k in range(args.warmup + args.steps):
        ev[0].record()
        pa.pa_swap_blocks(out_pairs, st.k_cache, st.v_cache, hk, hv, err=st.err)
        ev[1].record()
        pa.pa_swap_blocks(in_pairs, hk, hv, st.k_cache, st.v_cache, err=st.err)
        ev[2].record()
        if flat is not None:
            ev[3].record()
            link_host.copy_(flat[:link_host.numel()], non_blocking=True)
            ev[4].record()
        torch.cuda.synchronize()
        if k >= args.warmup:
            t_out.append(ev[0].elapsed_time(ev[1]))
            t_in.append(ev[1].elapsed_time(ev[2]))
            if flat is not None:
                t_link.append(ev[3].elapsed_time(ev[4]))
    flags = pa.pa_get_error(st.err)
    if flags:
        raise RuntimeError("kernel reported error bits 0x%x" % flags)
    gbs = lambda ms: nbytes / (ms * 1e-3) / 1e9
    out_gbs, in_gbs = gbs(statistics.mean(t_out)), gbs(statistics.mean(t_in))
    link = gbs(statistics.mean(t_link)) if t_link else None
    line = {
        "metric": "KV block swap GB/s (device pool <-> pinned host pool)", "value":
        round((out_gbs + in_gbs) / 2, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "dtype": st.k_cache.dtype.__repr__(),
        "data": "synthetic", "config": {"workload": wl.name, "blocks": n,
                                        "bytes_each_way": nbytes},
        "swap_out_gbs": round(out_gbs, 1), "swap_in_gbs": round(in_gbs, 1),
        "ms_out": round(statistics.mean(t_out), 4), "ms_in": round(statistics.mean(t_in), 4),
        "link_copy_gbs": None if link is None else round(link, 1),
        "link_copy": "one contiguous device -> pinned host copy of the same bytes (torch copy_)",
        "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)


def _seed(args):
    return DEFAULT_SEEDS[args.workload] if args.seed is None else args.seed


def _config(wl, args):
    return {
        "workload": wl.name, "num_seqs": wl.num_seqs, "q_heads": wl.num_q_heads,
        "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
        "kv_dtype": W.DTYPE_NAMES[W.FP8 if wl.fp8 else wl.dtype], "num_blocks": wl.num_blocks,
        "total_context_tokens": int(wl.seq_lens.sum()), "max_seq_len": wl.max_seq_len,
        "new_tokens_per_step": int(wl.new_seq.size), "copy_pairs": int(wl.copy_pairs.shape[0]),
        "window": wl.window,
        "seed": _seed(args), "recipe": wl.recipe,
        "l2": "flushed between timed steps: a %d MiB device buffer is written, then read" %
              (L2_FLUSH_BYTES >> 20),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3-8b-gqa", choices=sorted(W.CONFIGS))
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads of the oracle's CPU baseline (0: every available core)")
    ap.add_argument("--pool-blocks", type=int, default=None,
                    help="smaller pool for the Llama-3-8B workload (profiling captures)")
    ap.add_argument("--mode", default="step", choices=["step", "swap"],
                    help="step: the decode step (default); swap: block swap bandwidth")
    ap.add_argument("--swap-blocks", type=int, default=4096)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
        return
    if args.mode == "swap":
        run_swap(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    wl = res["wl"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, sample, _, n_cores = oracle_rate(wl, budget_s=args.cpu_baseline_seconds,
                                            threads=args.cpu_threads)
        cpu = {"value": round(r, 2), "unit": UNIT, "cores": n_cores, "kind": "oracle",
               "sample": sample}
    if rank == 0:
        value = job_throughput(wl.num_seqs, world, res["ms"])
        e2e = job_throughput(wl.num_seqs, world, res["e2e_ms"])
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 kv, f16 mma" if wl.fp8 else W.DTYPE_NAMES[wl.dtype],
            "data": "synthetic", "config": _config(wl, args),
            "roofline": res["roofline"], "cpu_baseline": cpu,
            "e2e": {"value": round(e2e, 1), "unit": UNIT, "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"], "ms_per_step": round(res["e2e_ms"], 4)},
            "gpu_launches": res["launches"] * world,
            "clocks": res["clocks"],
            "decode_ms": round(res["decode_ms"], 5),
            "step_algorithmic_bytes": res["bytes"]["step"],
            "step_gbs": round(res["bytes"]["step"] / (res["ms_local"] * 1e-3) / 1e9, 1),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
