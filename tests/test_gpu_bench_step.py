"""Every benchmark workload at full size, in the launch configuration the
benchmark times, against the oracle.

The step is built by bench.Step and captured as one CUDA graph, as the timed
loop replays it: copy-on-write pairs (shared-prefix workload), the slot
mapping and cache write in one launch, then the decode (or prefill) on the
default grid with the lengths and tables read before the grid-dependency
wait.  One replay is compared with the oracle: written cache rows and copied
blocks bit for bit, decode rows within the decode tolerance and within the
rounding bound of the oracle rounded once to the output dtype.  A second
replay of the same step must give the same output bits."""
import numpy as np
import pytest
import torch

import bench
import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import OracleState, check_parity

pytestmark = pytest.mark.gpu

# sequences the oracle evaluates where all of them would take too long on
# the host (None: every sequence)
SAMPLE = {"70b-long-context": [0, 7, 19, 31]}


def _bits(t):
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_cache(st, ref, wl):
    """The rows the step wrote and the blocks it copied, bit for bit."""
    nb, B, H, D = ref.k_cache.shape
    slots = ref.slots[ref.slots >= 0]
    for dev, host in ((st.k_cache, ref.k_cache), (st.v_cache, ref.v_cache)):
        flat_dev = dev.view(nb * B, H * D)
        got = _bits(flat_dev[torch.from_numpy(slots).to(dev.device)])
        assert np.array_equal(got, host.reshape(nb * B, H * D)[slots])
        if wl.copy_pairs.size:
            dst = np.ascontiguousarray(wl.copy_pairs[:, 1]).astype(np.int64)
            got = _bits(dev[torch.from_numpy(dst).to(dev.device)])
            assert np.array_equal(got, host[dst])


@pytest.mark.parametrize("name", [n for n in W.CONFIGS if n != "tiny"])
def test_bench_step_against_oracle(cuda_device, name):
    wl = W.CONFIGS[name](seed=bench.DEFAULT_SEEDS[name])
    st = bench.Step(wl, cuda_device)
    st.capture()
    st.g_step.replay()
    torch.cuda.synchronize()
    assert pa.pa_get_error(st.err) == 0
    first = st.out.clone()
    st.g_step.replay()
    torch.cuda.synchronize()
    assert pa.pa_get_error(st.err) == 0
    assert torch.equal(first.view(torch.int16), st.out.view(torch.int16))

    ref = OracleState(wl)
    ref.step()
    assert np.array_equal(st.slots.cpu().numpy(), ref.slots)
    _check_cache(st, ref, wl)

    flags = st.flags
    if wl.query_start is not None:
        # the rows of the sequences with the shortest and the longest prefix
        order = np.argsort(wl.seq_lens)
        for i in (int(order[0]), int(order[len(order) // 2]), int(order[-1])):
            q0, q1 = int(wl.query_start[i]), int(wl.query_start[i + 1])
            sub, sp = oracle.paged_prefill(wl.q[q0:q1], ref.k_cache, ref.v_cache, wl.dtype,
                                           wl.block_tables[i:i + 1], wl.seq_lens[i:i + 1],
                                           np.array([0, q1 - q0], np.int32), wl.scale,
                                           spread=True)
            check_parity(first[q0:q1], wl, sub, sp, "%s bench step, seq %d" % (name, i))
        return
    ids = SAMPLE.get(name)
    ids = np.arange(wl.num_seqs, dtype=np.int32) if ids is None else np.array(ids, np.int32)
    expected, spread = ref.decode(seq_ids=ids, spread=True)
    check_parity(first, wl, expected, spread, "%s bench step" % name, flags=flags, rows=ids)
