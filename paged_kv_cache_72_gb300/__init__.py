"""Paged KV-cache decode path for GB300 (sm_103a): a C-ABI CUDA library
(``libpa.so``, declared in ``include/pa.h``) and this thin Python binding.

The binding only marshals arguments (torch tensors -> device pointers, sizes
and the current CUDA stream); every step runs in the library's kernels.  There
is no fallback: if the library is missing, the calls raise.
"""
from ._lib import (PA_BF16, PA_DECODE_AUTO, PA_DECODE_MAX_CTAS, PA_DECODE_MMA, PA_DECODE_SIMT,
                   PA_DECODE_TABLES_READY, PA_DEVERR_BLOCK_ID, PA_DEVERR_COPY_PAIR,
                   PA_DEVERR_POSITION, PA_DEVERR_SEQ_LEN, PA_DEVERR_SLOT, PA_DEVERR_TIMEOUT,
                   PA_F16, PA_FP8_E4M3, PA_PREFILL_TENSOR_CORE, PA_PREFILL_WARP_MMA, PA_SWAP_IN,
                   PA_SWAP_OUT)
from .ops import (PAError, pa_cache_write, pa_cache_write_fp8, pa_cache_write_fp8_mapped, pa_cache_write_mapped, pa_copy_blocks, pa_decode,
                  pa_decode_fp8, pa_decode_window, pa_decode_workspace_size, pa_prefill, pa_prefill_kernel, pa_gather_kv, pa_get_error,
                  pa_slot_mapping, pa_swap_blocks, pa_version)

__all__ = [
    "PAError", "pa_slot_mapping", "pa_cache_write", "pa_cache_write_fp8", "pa_cache_write_fp8_mapped", "pa_cache_write_mapped", "pa_copy_blocks",
    "pa_decode", "pa_decode_fp8", "pa_decode_window", "pa_prefill", "pa_prefill_kernel",
    "pa_decode_workspace_size", "pa_gather_kv", "pa_get_error",
    "pa_version", "pa_swap_blocks", "PA_F16", "PA_BF16", "PA_FP8_E4M3",
    "PA_DECODE_AUTO", "PA_DECODE_SIMT", "PA_DECODE_MMA", "PA_DECODE_TABLES_READY",
    "PA_DECODE_MAX_CTAS", "PA_PREFILL_TENSOR_CORE", "PA_PREFILL_WARP_MMA", "PA_SWAP_OUT", "PA_SWAP_IN", "PA_DEVERR_SLOT", "PA_DEVERR_BLOCK_ID",
    "PA_DEVERR_SEQ_LEN", "PA_DEVERR_COPY_PAIR", "PA_DEVERR_TIMEOUT", "PA_DEVERR_POSITION",
]
