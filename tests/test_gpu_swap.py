"""Block swap between the GPU pool and a pinned host pool ("vLLM anatomy",
section "Memory Pressure and Preemption": swapping moves physical blocks to the
CPU's memory and back).  Bit-exact against the oracle's block copy; a
sequence swapped out and back into other blocks decodes to the same bits
through its remapped table; E4M3 pools; bad pairs are reported, not copied;
pageable host memory is refused."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState

pytestmark = pytest.mark.gpu


def _host_pool(like, n):
    return torch.zeros((n,) + tuple(like.shape[1:]), dtype=like.dtype).pin_memory()


def _np(t):
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype != torch.uint8 else t.numpy()


@pytest.mark.parametrize("fp8", [False, True])
def test_swap_out_and_back_in(cuda_device, fp8):
    wl = W.random_workload(111, W.BF16, 8, 2, 128, 16, [40, 300, 5], num_blocks=64,
                           fp8_scales=(2.0 ** -6, 2.0 ** -6) if fp8 else None)
    st = GpuState(wl)
    used = np.unique(wl.block_tables[wl.block_tables >= 0]).astype(np.int32)
    hk, hv = _host_pool(st.k_cache, 40), _host_pool(st.v_cache, 40)
    out_pairs = np.stack([used, 39 - np.arange(used.size)], axis=1).astype(np.int32)
    pa.pa_swap_blocks(torch.from_numpy(out_pairs).cuda(), st.k_cache, st.v_cache, hk, hv,
                      err=st.err)
    torch.cuda.synchronize()
    ek = np.zeros_like(_np(hk))
    ev = np.zeros_like(ek)
    oracle.swap_blocks(wl.k_cache, wl.v_cache, ek, ev, out_pairs)
    assert np.array_equal(_np(hk), ek) and np.array_equal(_np(hv), ev)
    # back in, into blocks the sequences did not use, then decode through the
    # remapped table: the same bits as before
    free = np.setdiff1d(np.arange(wl.num_blocks), used)[:used.size].astype(np.int32)
    in_pairs = np.stack([39 - np.arange(used.size), free], axis=1).astype(np.int32)
    kc2 = torch.zeros_like(st.k_cache)
    vc2 = torch.zeros_like(st.v_cache)
    pa.pa_swap_blocks(torch.from_numpy(in_pairs).cuda(), hk, hv, kc2, vc2, err=st.err)
    remap = np.full(wl.num_blocks, -1, np.int32)
    remap[used] = free
    bt2 = np.where(wl.block_tables >= 0, remap[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    bt2 = torch.from_numpy(bt2).cuda()
    if fp8:
        a = pa.pa_decode_fp8(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                             wl.scale, wl.k_scale, wl.v_scale)
        b = pa.pa_decode_fp8(st.q, kc2, vc2, bt2, st.seq_lens, wl.scale, wl.k_scale, wl.v_scale)
    else:
        a = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale)
        b = pa.pa_decode(st.q, kc2, vc2, bt2, st.seq_lens, wl.scale)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert pa.pa_get_error(st.err) == 0


def test_swap_reports_bad_pairs(cuda_device):
    wl = W.random_workload(112, W.F16, 4, 4, 64, 8, [20], num_blocks=8)
    st = GpuState(wl)
    hk, hv = _host_pool(st.k_cache, 4), _host_pool(st.v_cache, 4)
    bad = torch.tensor([[0, 4], [1, 1], [2, 1], [9, 0]], dtype=torch.int32).cuda()
    pa.pa_swap_blocks(bad, st.k_cache, st.v_cache, hk, hv, err=st.err)
    assert pa.pa_get_error(st.err) == pa.PA_DEVERR_COPY_PAIR
    assert not hk.any() and not hv.any()


def test_swap_with_pageable_host_memory_copies_or_refuses(cuda_device):
    # where the GPU reads pageable host memory (a Grace-Blackwell node) the swap
    # goes through; elsewhere the library refuses it with PA_ERR_INVALID_ARG
    wl = W.random_workload(113, W.BF16, 4, 4, 64, 8, [20], num_blocks=8)
    st = GpuState(wl)
    hk = torch.zeros((4,) + tuple(st.k_cache.shape[1:]), dtype=st.k_cache.dtype)
    hv = torch.zeros_like(hk)
    pairs = torch.tensor([[1, 0], [2, 3]], dtype=torch.int32).cuda()
    try:
        pa.pa_swap_blocks(pairs, st.k_cache, st.v_cache, hk, hv, err=st.err)
    except pa.PAError as e:
        assert e.status == 1
        return
    torch.cuda.synchronize()
    assert torch.equal(hk[0], st.k_cache[1].cpu()) and torch.equal(hv[3], st.v_cache[2].cpu())
    assert not hk[1].any() and not hk[2].any()
    assert pa.pa_get_error(st.err) == 0
