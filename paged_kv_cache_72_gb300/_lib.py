"""ctypes declarations of the C ABI in include/pa.h.

Loading fails loudly: there is no fallback implementation of any entry point.
"""
import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")

# status codes and flags, mirrored from include/pa.h
PA_F16 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2
PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_INDEX = 5
PA_DEVERR_SLOT = 0x1
PA_DEVERR_BLOCK_ID = 0x2
PA_DEVERR_SEQ_LEN = 0x4
PA_DEVERR_COPY_PAIR = 0x8
PA_DEVERR_TIMEOUT = 0x10
PA_DEVERR_POSITION = 0x20
PA_SWAP_OUT = 0
PA_SWAP_IN = 1
PA_DECODE_AUTO = 0
PA_DECODE_SIMT = 1
PA_DECODE_MMA = 2
PA_DECODE_TABLES_READY = 0x100
PA_NOALLOC_SCRATCH_BYTES = 16 << 20
PA_DECODE_MAX_CTAS = 16384
PA_PREFILL_WARP_MMA = 0
PA_PREFILL_TENSOR_CORE = 1

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/pa.h
SIGNATURES = {
    "pa_slot_mapping": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp]),
    "pa_cache_write": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _i32, _i32, _i32, _i32,
                                      _vp, _vp]),
    "pa_cache_write_mapped": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _i64, _vp, _vp,
                                             _i64, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "pa_copy_blocks": (ctypes.c_int, [_vp, _i32, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _vp, _vp]),
    "pa_swap_blocks": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _i64, _vp, _vp, _i64, _i32, _i32,
                                      _i32, _i32, _vp, _vp]),
    "pa_cache_write_fp8": (ctypes.c_int, [_vp, _vp, _i32, _vp, _i64, _vp, _vp, _i64, _i32, _i32,
                                          _i32, ctypes.c_float, ctypes.c_float, _vp, _vp]),
    "pa_cache_write_fp8_mapped": (ctypes.c_int, [_vp, _vp, _i32, _vp, _i32, _i32, _vp, _vp, _i64,
                                                 _vp, _vp, _i64, _i32, _i32, _i32, ctypes.c_float,
                                                 ctypes.c_float, _vp, _vp, _vp]),
    "pa_decode_workspace_size": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                                ctypes.POINTER(_sz)]),
    "pa_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i64,
                                 _i32, ctypes.c_float, _vp, _vp, _sz, _i32, _i32, _vp, _vp]),
    "pa_decode_window": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                        _i32, _i64, _i32, ctypes.c_float, _i32, _vp, _vp, _sz,
                                        _i32, _i32, _vp, _vp]),
    "pa_decode_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                     _i64, _i32, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                     _vp, _vp, _sz, _i32, _i32, _vp, _vp]),
    "pa_prefill_workspace_size": (ctypes.c_int, [ctypes.POINTER(_sz)]),
    "pa_prefill_kernel": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, _i32,
                                         ctypes.POINTER(_i32)]),
    "pa_prefill": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                                  _i32, _i64, _i32, ctypes.c_float, _vp, _vp, _sz, _vp, _vp]),
    "pa_decode_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                         _i32, _i64, _i32, ctypes.c_float, _vp, _i32, _i32, _vp,
                                         _vp]),
    "pa_gather_kv": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i64,
                                    _i32, _i32, _vp, _vp, _vp, _vp]),
    "pa_get_error": (ctypes.c_int, [_vp, _vp, ctypes.POINTER(_i32)]),
    "pa_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "pa_version": (ctypes.c_int, []),
}

_handle = None


def load(path=LIB_PATH):
    """Load libpa.so and declare every entry point.  Raises if it is missing."""
    global _handle
    if _handle is None:
        if not os.path.exists(path):
            raise ImportError(
                "libpa.so is not built (%s); run paged_kv_cache_72_gb300.build.build()" % path)
        h = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _handle = h
    return _handle
