"""Scalar CPU oracle for MXFP8 / NVFP4 block-scaled quantization.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (``fp4_quantization_gb300``) never does, and this package
imports nothing from it.

The arithmetic lives in ``mxq_oracle.c`` (plain C99, one IEEE operation per
step); this module only marshals numpy arrays into it.  Inputs are bf16 bit
patterns held in ``numpy.uint16`` arrays; a 2-D view with a unit inner stride
is accepted as is, so a window of a large matrix can be checked without a copy.
"""
import ctypes
import numpy as np

from . import build as _build

ROWWISE, COLWISE, DBIAS = 1, 2, 4
NVFP4_2D = 16
SCALE_RCEIL = 64
ACT_NONE, ACT_GELU_TANH, ACT_SILU = 0, 1, 2

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        L.orc_bf16_decode.restype = ctypes.c_double
        L.orc_bf16_decode.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_double]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e8m0_code.restype = ctypes.c_uint8
        L.orc_e8m0_code.argtypes = [ctypes.c_double]
        for name in ("orc_e4m3_encode_array", "orc_e2m1_encode_array", "orc_e8m0_code_array",
                     "orc_e8m0_code_rceil_array"):
            fn = getattr(L, name)
            fn.restype = None
            fn.argtypes = [dp, i64, u8p]
        L.orc_gelu_tanh.restype = ctypes.c_float
        L.orc_gelu_tanh.argtypes = [ctypes.c_float]
        L.orc_swiglu.restype = ctypes.c_float
        L.orc_swiglu.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_geglu.restype = ctypes.c_float
        L.orc_geglu.argtypes = [ctypes.c_float, ctypes.c_float]
        for name in ("orc_dgelu_tanh", "orc_dsilu"):
            getattr(L, name).restype = ctypes.c_float
            getattr(L, name).argtypes = [ctypes.c_float]
        L.orc_mx_quantize_gated.restype = ctypes.c_int
        L.orc_mx_quantize_gated.argtypes = [ctypes.c_void_p, i64, i64, i64, i64, ctypes.c_int,
                                            ctypes.c_int, u8p, u8p, u8p, u8p]
        L.orc_mx_quantize_dact.restype = ctypes.c_int
        L.orc_mx_quantize_dact.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, i64, i64, i64,
                                           ctypes.c_int, ctypes.c_int, u8p, u8p, u8p, u8p, f32p]
        L.orc_mx_quantize_dgated.restype = ctypes.c_int
        L.orc_mx_quantize_dgated.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, i64, i64, i64,
                                             i64, ctypes.c_int, ctypes.c_int, u8p, u8p, u8p, u8p]
        L.orc_mx_quantize.restype = ctypes.c_int
        L.orc_mx_quantize.argtypes = [ctypes.c_void_p, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                      u8p, u8p, u8p, u8p, f32p]
        L.orc_mx_quantize_swiglu.restype = ctypes.c_int
        L.orc_mx_quantize_swiglu.argtypes = [ctypes.c_void_p, i64, i64, i64, i64, ctypes.c_int,
                                             u8p, u8p, u8p, u8p]
        L.orc_bf16_amax.restype = ctypes.c_float
        L.orc_bf16_amax.argtypes = [ctypes.c_void_p, i64, i64, i64]
        L.orc_nvfp4_quantize.restype = ctypes.c_int
        L.orc_nvfp4_quantize.argtypes = [ctypes.c_void_p, i64, i64, i64, ctypes.c_float,
                                         ctypes.c_int, f32p, u8p, u8p, u8p, u8p]
        _lib = L
    return _lib


def _u8(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _f32(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _matrix(x):
    """Return (pointer, rows, cols, row stride in elements) of a uint16 view."""
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError("oracle input must be a 2-D numpy.uint16 array of bf16 bit patterns")
    if x.size == 0:
        return ctypes.c_void_p(x.ctypes.data), x.shape[0], x.shape[1], x.shape[1]
    if x.shape[1] > 1 and x.strides[1] != 2:
        raise ValueError("oracle input needs a unit inner stride")
    ld = x.strides[0] // 2 if x.shape[0] > 1 else x.shape[1]
    return ctypes.c_void_p(x.ctypes.data), x.shape[0], x.shape[1], ld


# --------------------------------------------------------------------------
# Scalar / elementwise helpers
# --------------------------------------------------------------------------

def e4m3_encode(v):
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e4m3_encode_array(v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), v.size, _u8(out))
    return out


def e2m1_encode(v):
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e2m1_encode_array(v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), v.size, _u8(out))
    return out


def e8m0_code(amax):
    v = np.ascontiguousarray(amax, dtype=np.float64).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e8m0_code_array(v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), v.size, _u8(out))
    return out


def e8m0_code_rceil(amax):
    v = np.ascontiguousarray(amax, dtype=np.float64).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e8m0_code_rceil_array(v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), v.size,
                                    _u8(out))
    return out


def e4m3_decode(code):
    return lib().orc_e4m3_decode(int(code))


def e2m1_decode(code):
    return lib().orc_e2m1_decode(int(code))


def bf16_decode(bits):
    return lib().orc_bf16_decode(int(bits))


def gelu_tanh(x):
    return float(lib().orc_gelu_tanh(float(x)))


def swiglu(g, u):
    return float(lib().orc_swiglu(float(g), float(u)))


def geglu(g, u):
    return float(lib().orc_geglu(float(g), float(u)))


def dgelu_tanh(x):
    return float(lib().orc_dgelu_tanh(float(x)))


def dsilu(x):
    return float(lib().orc_dsilu(float(x)))


# --------------------------------------------------------------------------
# Whole-matrix quantizers
# --------------------------------------------------------------------------

def mx_quantize(x, flags=ROWWISE | COLWISE, act=ACT_NONE):
    """MXFP8 quantization of bf16 bits x[M, K].  Returns a dict with the
    requested outputs: q_row [M,K], s_row [M,K/32], q_col [K,M],
    s_col [K,M/32] (uint8) and dbias [K] (float32)."""
    p, M, K, ld = _matrix(x)
    out = {}
    if flags & ROWWISE:
        out["q_row"] = np.empty((M, K), np.uint8)
        out["s_row"] = np.empty((M, K // 32), np.uint8)
    if flags & COLWISE:
        out["q_col"] = np.empty((K, M), np.uint8)
        out["s_col"] = np.empty((K, M // 32), np.uint8)
    if flags & DBIAS:
        out["dbias"] = np.empty(K, np.float32)
    rc = lib().orc_mx_quantize(p, M, K, ld, flags & ~SCALE_SWIZZLED, act,
                               _u8(out.get("q_row")), _u8(out.get("s_row")),
                               _u8(out.get("q_col")), _u8(out.get("s_col")),
                               _f32(out.get("dbias")))
    if rc != 0:
        raise ValueError(f"orc_mx_quantize rejected M={M} K={K} ld={ld} act={act}")
    return _maybe_swizzle(out, flags)


def mx_quantize_swiglu(x, N, up_offset=None, flags=ROWWISE | COLWISE):
    """SwiGLU-gated MXFP8: y = silu(x[:, :N]) * x[:, up_offset:up_offset+N]
    (up_offset defaults to N), quantized rowwise/colwise like mx_quantize."""
    p, M, W, ld = _matrix(x)
    if up_offset is None:
        up_offset = N
    out = {}
    if flags & ROWWISE:
        out["q_row"] = np.empty((M, N), np.uint8)
        out["s_row"] = np.empty((M, N // 32), np.uint8)
    if flags & COLWISE:
        out["q_col"] = np.empty((N, M), np.uint8)
        out["s_col"] = np.empty((N, M // 32), np.uint8)
    rc = lib().orc_mx_quantize_swiglu(p, M, N, ld, up_offset, flags,
                                      _u8(out.get("q_row")), _u8(out.get("s_row")),
                                      _u8(out.get("q_col")), _u8(out.get("s_col")))
    if rc != 0:
        raise ValueError(f"orc_mx_quantize_swiglu rejected M={M} N={N} ld={ld}")
    return out


def bf16_amax(x):
    p, M, K, ld = _matrix(x)
    return float(lib().orc_bf16_amax(p, M, K, ld))


def nvfp4_quantize(x, tensor_amax=None, flags=ROWWISE | COLWISE):
    """NVFP4 quantize-transpose of bf16 bits x[M, K] given the tensor amax
    (computed over x when None).  Returns global_scale (float), q_row
    [M,K/2], s_row [M,K/16], q_t [K,M/2], s_t [K,M/16].  flags | NVFP4_2D
    takes one scale per 16x16 block."""
    p, M, K, ld = _matrix(x)
    if tensor_amax is None:
        tensor_amax = bf16_amax(x)
    out = {}
    if flags & ROWWISE:
        out["q_row"] = np.empty((M, K // 2), np.uint8)
        out["s_row"] = np.empty((M, K // 16), np.uint8)
    if flags & COLWISE:
        out["q_t"] = np.empty((K, M // 2), np.uint8)
        out["s_t"] = np.empty((K, M // 16), np.uint8)
    g = np.zeros(1, np.float32)
    rc = lib().orc_nvfp4_quantize(p, M, K, ld, float(tensor_amax), flags, _f32(g),
                                  _u8(out.get("q_row")), _u8(out.get("s_row")),
                                  _u8(out.get("q_t")), _u8(out.get("s_t")))
    if rc != 0:
        raise ValueError(f"orc_nvfp4_quantize rejected M={M} K={K} ld={ld}")
    out["global_scale"] = float(g[0])
    return out


def _mx_outputs(M, K, flags):
    out = {}
    if flags & ROWWISE:
        out["q_row"] = np.empty((M, K), np.uint8)
        out["s_row"] = np.empty((M, K // 32), np.uint8)
    if flags & COLWISE:
        out["q_col"] = np.empty((K, M), np.uint8)
        out["s_col"] = np.empty((K, M // 32), np.uint8)
    if flags & DBIAS:
        out["dbias"] = np.empty(K, np.float32)
    return out


def mx_quantize_gated(x, N, act=ACT_SILU, up_offset=None, flags=ROWWISE | COLWISE):
    """Gated MXFP8: y = act(x[:, :N]) * x[:, up_offset:up_offset+N] with act
    ACT_SILU (SwiGLU) or ACT_GELU_TANH (GeGLU); outputs as mx_quantize."""
    p, M, W, ld = _matrix(x)
    if up_offset is None:
        up_offset = N
    out = _mx_outputs(M, N, flags & (ROWWISE | COLWISE))
    rc = lib().orc_mx_quantize_gated(p, M, N, ld, up_offset, flags & ~SCALE_SWIZZLED, act,
                                     _u8(out.get("q_row")), _u8(out.get("s_row")),
                                     _u8(out.get("q_col")), _u8(out.get("s_col")))
    if rc != 0:
        raise ValueError(f"orc_mx_quantize_gated rejected M={M} N={N} ld={ld} act={act}")
    return _maybe_swizzle(out, flags)


def mx_quantize_dact(grad, x, act, flags=ROWWISE | COLWISE):
    """Backward MXFP8: y = grad * act'(x) (act ACT_GELU_TANH or ACT_SILU),
    quantized like mx_quantize; flags | DBIAS adds the column sums of y."""
    pg, M, K, ldg = _matrix(grad)
    px, M2, K2, ldx = _matrix(x)
    if (M2, K2) != (M, K):
        raise ValueError("grad and x shapes differ")
    out = _mx_outputs(M, K, flags)
    rc = lib().orc_mx_quantize_dact(pg, px, M, K, ldg, ldx, flags & ~SCALE_SWIZZLED, act,
                                    _u8(out.get("q_row")), _u8(out.get("s_row")),
                                    _u8(out.get("q_col")), _u8(out.get("s_col")),
                                    _f32(out.get("dbias")))
    if rc != 0:
        raise ValueError(f"orc_mx_quantize_dact rejected M={M} K={K} act={act}")
    return _maybe_swizzle(out, flags)


def mx_quantize_dgated(grad, x, N, act, up_offset=None, flags=ROWWISE | COLWISE):
    """Backward gated MXFP8: grad [M, N], x = [gate | up]; y [M, 2N] =
    [grad * up * act'(gate) | grad * act(gate)], quantized like mx_quantize."""
    pg, M, Ng, ldg = _matrix(grad)
    px, M2, W, ldx = _matrix(x)
    if up_offset is None:
        up_offset = N
    if M2 != M or Ng != N:
        raise ValueError("grad must be [M, N] for x = [gate | up]")
    out = _mx_outputs(M, 2 * N, flags & (ROWWISE | COLWISE))
    rc = lib().orc_mx_quantize_dgated(pg, px, M, N, ldg, ldx, up_offset, flags & ~SCALE_SWIZZLED,
                                      act,
                                      _u8(out.get("q_row")), _u8(out.get("s_row")),
                                      _u8(out.get("q_col")), _u8(out.get("s_col")))
    if rc != 0:
        raise ValueError(f"orc_mx_quantize_dgated rejected M={M} N={N} act={act}")
    return _maybe_swizzle(out, flags)


# --------------------------------------------------------------------------
# Tiled scale layout (flag SCALE_SWIZZLED of the MXFP8 calls)
# --------------------------------------------------------------------------

SCALE_SWIZZLED = 128


def _maybe_swizzle(out, flags):
    if flags & SCALE_SWIZZLED:
        for key in ("s_row", "s_col"):
            if key in out:
                out[key] = swizzle_scales(out[key])
    return out


def swizzled_shape(R, C):
    """Padded [R', C'] of an [R][C] scale matrix in the tiled layout."""
    return -(-R // 128) * 128, -(-C // 4) * 4


def swizzle_scales(s):
    """[R][C] row-major scale bytes -> the tiled layout block-scaled GEMMs
    read: padded to R' = ceil(R/128)*128 rows and C' = ceil(C/4)*4 columns
    (padding 0), cut into 128x4 tiles stored one after another in row-major
    tile order (tile (i, j) at byte (i * C'/4 + j) * 512); inside a tile,
    entry (r, c) sits at byte (r % 32) * 16 + (r // 32) * 4 + c.  Returned
    as an [R', C'] uint8 array holding those bytes in order."""
    s = np.asarray(s, dtype=np.uint8)
    R, C = s.shape
    Rp, Cp = swizzled_shape(R, C)
    out = np.zeros(Rp * Cp, np.uint8)
    tiles_c = Cp // 4
    for r in range(R):
        i, rr = divmod(r, 128)
        for c in range(C):
            j, cc = divmod(c, 4)
            out[(i * tiles_c + j) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc] = s[r, c]
    return out.reshape(Rp, Cp)
