"""ctypes loader for libmxq.so.

The library is built in-tree by ``fp4_quantization_gb300/build.py`` (called
from ``__graft_entry__.build()``).  Loading it needs no GPU; calling into it
does.  A missing or unloadable library raises ImportError: there is no
fallback implementation.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmxq.so")

# Every exported entry point with (restype, argtypes); kept in the order of
# include/mxq.h.
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_sz = ctypes.c_size_t
SIGNATURES = {
    "mxq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mxq_workspace_bytes": (_sz, [ctypes.c_int, _i64, _i64, _u32]),
    "mx_quantize_rowcol": (ctypes.c_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp, _vp, _vp, _vp,
                                          _vp, _sz, _vp, _vp]),
    "mx_quantize_rowcol_dbias_noalloc": (ctypes.c_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp,
                                                        _vp, _vp, _vp, _vp, _vp]),
    "mx_quantize_rowcol_host": (ctypes.c_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp, _vp, _vp,
                                               _vp, _sz, _vp]),
    "mx_quantize_gated": (ctypes.c_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp, _vp, _vp, _vp,
                                         _vp]),
    "mx_quantize_dact": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i64, _i64, _u32, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _sz, _vp, _vp]),
    "mx_quantize_dgated": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i64, _i64, _u32, _vp, _vp, _vp,
                                          _vp, _vp, _vp]),
    "bf16_amax": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp]),
    "nvfp4_quantize_transpose": (ctypes.c_int, [_vp, _i64, _i64, _i64, _u32, _vp, _vp, _vp, _vp,
                                                _vp, _vp, _vp, _sz, _vp, _vp]),
    "mxq_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint64, _vp, _vp]),
}

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (needs nvcc); there is no fallback implementation")
        try:
            L = ctypes.CDLL(LIB_PATH)
        except OSError as e:
            raise ImportError(f"cannot load {LIB_PATH}: {e}") from e
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


lib()
