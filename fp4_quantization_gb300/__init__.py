"""GB300 (sm_103a) block-scaled quantization: bf16 -> MXFP8 / NVFP4.

Thin Python binding over libmxq.so, whose C ABI is declared in
``include/mxq.h``.  The functions here carry the same names as the C entry
points and only marshal arguments: they allocate outputs with torch when the
caller does not pass them, pass raw device pointers and the current CUDA
stream, and raise ``MxqError`` on a non-zero status.  Every step of the
quantization runs in the library's kernels; there is no fallback path, and
importing this package fails if libmxq.so cannot be loaded.
"""
import ctypes

import torch

from . import _lib

ROWWISE = 1
COLWISE = 2
DBIAS = 4
ACT_GELU_TANH = 8
NVFP4_2D = 16
ACT_SILU = 32
SCALE_RCEIL = 64
SCALE_SWIZZLED = 128


def scale_shape(R, C, flags):
    """Shape of an [R][C] scale matrix as written under `flags`: padded to
    128 x 4 tiles with SCALE_SWIZZLED, else [R, C]."""
    if flags & SCALE_SWIZZLED:
        return (-(-R // 128) * 128, -(-C // 4) * 4)
    return (R, C)
OP_ROWCOL = 0
OP_NVFP4 = 1
OP_DACT = 2
OP_ROWCOL_HOST = 3
DEVERR_TIMEOUT = 1

STATUS_NAMES = {0: "MXQ_OK", 1: "MXQ_EINVAL", 2: "MXQ_ESHAPE", 3: "MXQ_EALIGN",
                4: "MXQ_EARCH", 5: "MXQ_EWORKSPACE", 6: "MXQ_ECUDA"}


class MxqError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.lib().mxq_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def library_path():
    return _lib.LIB_PATH


def _check(status, where):
    if status != 0:
        raise MxqError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _input(x, name="x"):
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or x.dim() != 2:
        raise TypeError(f"{name} must be a 2-D torch.bfloat16 tensor")
    if not x.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if x.size(1) > 1 and x.stride(1) != 1:
        raise ValueError(f"{name} needs a unit column stride")
    return x.stride(0) if x.size(0) > 1 else x.size(1)


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def mxq_workspace_bytes(op, M, K, flags):
    return int(_lib.lib().mxq_workspace_bytes(op, M, K, flags))


def mx_quantize_rowcol(x, flags=ROWWISE | COLWISE, *, q_row=None, s_row=None, q_col=None,
                       s_col=None, dbias=None, workspace=None, dev_err=None, stream=None):
    """bf16 x[M, K] -> MXFP8.  Returns a dict with q_row [M,K] / s_row
    [M,K/32] (ROWWISE), q_col [K,M] / s_col [K,M/32] (COLWISE), dbias [K]
    fp32 (DBIAS); codes and scales are torch.uint8."""
    ldx = _input(x)
    M, K = x.shape
    dev = x.device
    out = {}
    if flags & ROWWISE:
        out["q_row"] = q_row if q_row is not None else _empty((M, K), torch.uint8, dev)
        out["s_row"] = s_row if s_row is not None else _empty(scale_shape(M, K // 32, flags),
                                                              torch.uint8, dev)
    if flags & COLWISE:
        out["q_col"] = q_col if q_col is not None else _empty((K, M), torch.uint8, dev)
        out["s_col"] = s_col if s_col is not None else _empty(scale_shape(K, M // 32, flags),
                                                              torch.uint8, dev)
    ws_bytes = 0
    if flags & DBIAS:
        out["dbias"] = dbias if dbias is not None else _empty((K,), torch.float32, dev)
        if workspace is None:
            need = mxq_workspace_bytes(OP_ROWCOL, M, K, flags)
            workspace = _empty((max(need, 16),), torch.uint8, dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.lib().mx_quantize_rowcol(
        _ptr(x), M, K, ldx, flags, _ptr(out.get("q_row")), _ptr(out.get("s_row")),
        _ptr(out.get("q_col")), _ptr(out.get("s_col")), _ptr(out.get("dbias")),
        _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    _check(st, "mx_quantize_rowcol")
    return out


def mx_quantize_rowcol_dbias_noalloc(x, flags=ROWWISE | COLWISE, *, q_row=None, s_row=None,
                                     q_col=None, s_col=None, dbias=None, dev_err=None,
                                     stream=None):
    """mx_quantize_rowcol with dbias, for callers that cannot allocate a
    workspace: the library keeps the band sums in its own fixed 8 MiB
    device array (see include/mxq.h for the limit, and for ordering calls
    that share it).  Outputs not passed in are allocated here with torch,
    as in the other bindings; pass them all to allocate nothing."""
    ldx = _input(x)
    M, K = x.shape
    dev = x.device
    out = {}
    if flags & ROWWISE:
        out["q_row"] = q_row if q_row is not None else _empty((M, K), torch.uint8, dev)
        out["s_row"] = s_row if s_row is not None else _empty(scale_shape(M, K // 32, flags),
                                                              torch.uint8, dev)
    if flags & COLWISE:
        out["q_col"] = q_col if q_col is not None else _empty((K, M), torch.uint8, dev)
        out["s_col"] = s_col if s_col is not None else _empty(scale_shape(K, M // 32, flags),
                                                              torch.uint8, dev)
    out["dbias"] = dbias if dbias is not None else _empty((K,), torch.float32, dev)
    st = _lib.lib().mx_quantize_rowcol_dbias_noalloc(
        _ptr(x), M, K, ldx, flags, _ptr(out.get("q_row")), _ptr(out.get("s_row")),
        _ptr(out.get("q_col")), _ptr(out.get("s_col")), _ptr(out["dbias"]), _ptr(dev_err),
        _stream(stream))
    _check(st, "mx_quantize_rowcol_dbias_noalloc")
    return out


def mx_quantize_rowcol_host(x, flags=ROWWISE | COLWISE, *, q_row=None, s_row=None, q_col=None,
                            s_col=None, workspace=None, stream=None):
    """mx_quantize_rowcol of a bf16 matrix in host memory: outputs in host
    memory (page-locked when allocated here), computed by panels pipelined
    through the device.  Returns once the work is enqueued; synchronise the
    stream before reading the outputs."""
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or x.dim() != 2:
        raise TypeError("x must be a 2-D torch.bfloat16 tensor")
    if x.is_cuda:
        raise TypeError("x must be in host memory (use mx_quantize_rowcol for device tensors)")
    if x.size(1) > 1 and x.stride(1) != 1:
        raise ValueError("x needs a unit column stride")
    M, K = x.shape
    ldx = x.stride(0) if M > 1 else K

    def host(shape, given):
        return given if given is not None else torch.empty(shape, dtype=torch.uint8).pin_memory()

    out = {}
    if flags & ROWWISE:
        out["q_row"] = host((M, K), q_row)
        out["s_row"] = host(scale_shape(M, K // 32, flags), s_row)
    if flags & COLWISE:
        out["q_col"] = host((K, M), q_col)
        out["s_col"] = host(scale_shape(K, M // 32, flags), s_col)
    if workspace is None:
        need = mxq_workspace_bytes(OP_ROWCOL_HOST, M, K, flags)
        workspace = _empty((max(need, 256),), torch.uint8, torch.device("cuda"))
    st = _lib.lib().mx_quantize_rowcol_host(
        _ptr(x), M, K, ldx, flags, _ptr(out.get("q_row")), _ptr(out.get("s_row")),
        _ptr(out.get("q_col")), _ptr(out.get("s_col")), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "mx_quantize_rowcol_host")
    return out


def mx_quantize_gated(x, flags=ROWWISE | COLWISE, *, q_row=None, s_row=None, q_col=None,
                      s_col=None, dev_err=None, stream=None):
    """Gated MXFP8 of x[M, 2N] = [gate | up]; y = silu(gate) * up (SwiGLU,
    the default) or gelu_tanh(gate) * up (flags | ACT_GELU_TANH: GeGLU) in
    fp32, quantized like mx_quantize_rowcol (outputs sized by N)."""
    ldx = _input(x)
    M, W = x.shape
    if W % 2:
        raise ValueError("x must hold [gate | up] halves of equal width")
    N = W // 2
    dev = x.device
    out = {}
    if flags & ROWWISE:
        out["q_row"] = q_row if q_row is not None else _empty((M, N), torch.uint8, dev)
        out["s_row"] = s_row if s_row is not None else _empty(scale_shape(M, N // 32, flags),
                                                              torch.uint8, dev)
    if flags & COLWISE:
        out["q_col"] = q_col if q_col is not None else _empty((N, M), torch.uint8, dev)
        out["s_col"] = s_col if s_col is not None else _empty(scale_shape(N, M // 32, flags),
                                                              torch.uint8, dev)
    st = _lib.lib().mx_quantize_gated(
        _ptr(x), M, N, ldx, flags, _ptr(out.get("q_row")), _ptr(out.get("s_row")),
        _ptr(out.get("q_col")), _ptr(out.get("s_col")), _ptr(dev_err), _stream(stream))
    _check(st, "mx_quantize_gated")
    return out


def _mx_outputs(M, K, flags, dev, q_row, s_row, q_col, s_col):
    out = {}
    if flags & ROWWISE:
        out["q_row"] = q_row if q_row is not None else _empty((M, K), torch.uint8, dev)
        out["s_row"] = s_row if s_row is not None else _empty(scale_shape(M, K // 32, flags),
                                                              torch.uint8, dev)
    if flags & COLWISE:
        out["q_col"] = q_col if q_col is not None else _empty((K, M), torch.uint8, dev)
        out["s_col"] = s_col if s_col is not None else _empty(scale_shape(K, M // 32, flags),
                                                              torch.uint8, dev)
    return out


def mx_quantize_dact(grad, x, flags, *, q_row=None, s_row=None, q_col=None, s_col=None,
                     dbias=None, workspace=None, dev_err=None, stream=None):
    """Backward MXFP8: y = grad * act'(x) for grad, x [M, K] bf16, with act
    gelu_tanh (flags | ACT_GELU_TANH) or silu (flags | ACT_SILU); outputs as
    mx_quantize_rowcol, dbias = column sums of y with DBIAS."""
    ldg = _input(grad, "grad")
    ldx = _input(x)
    M, K = x.shape
    if tuple(grad.shape) != (M, K):
        raise ValueError("grad and x shapes differ")
    dev = x.device
    out = _mx_outputs(M, K, flags, dev, q_row, s_row, q_col, s_col)
    ws_bytes = 0
    if flags & DBIAS:
        out["dbias"] = dbias if dbias is not None else _empty((K,), torch.float32, dev)
        if workspace is None:
            need = mxq_workspace_bytes(OP_DACT, M, K, flags)
            workspace = _empty((max(need, 16),), torch.uint8, dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.lib().mx_quantize_dact(
        _ptr(grad), _ptr(x), M, K, ldg, ldx, flags, _ptr(out.get("q_row")),
        _ptr(out.get("s_row")), _ptr(out.get("q_col")), _ptr(out.get("s_col")),
        _ptr(out.get("dbias")), _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    _check(st, "mx_quantize_dact")
    return out


def mx_quantize_dgated(grad, x, flags=ROWWISE | COLWISE, *, q_row=None, s_row=None, q_col=None,
                       s_col=None, dev_err=None, stream=None):
    """Backward of the gated activation: grad [M, N], x [M, 2N] = [gate |
    up]; y [M, 2N] = [grad * up * act'(gate) | grad * act(gate)] with act
    silu (default) or gelu_tanh (flags | ACT_GELU_TANH), quantized like
    mx_quantize_rowcol (outputs sized by 2N)."""
    ldg = _input(grad, "grad")
    ldx = _input(x)
    M, W = x.shape
    if W % 2 or tuple(grad.shape) != (M, W // 2):
        raise ValueError("x must be [M, 2N] = [gate | up] and grad [M, N]")
    N = W // 2
    out = _mx_outputs(M, W, flags, x.device, q_row, s_row, q_col, s_col)
    st = _lib.lib().mx_quantize_dgated(
        _ptr(grad), _ptr(x), M, N, ldg, ldx, flags, _ptr(out.get("q_row")),
        _ptr(out.get("s_row")), _ptr(out.get("q_col")), _ptr(out.get("s_col")), _ptr(dev_err),
        _stream(stream))
    _check(st, "mx_quantize_dgated")
    return out


def bf16_amax(x, *, out=None, stream=None):
    """Largest |x| as a 1-element fp32 device tensor."""
    ldx = _input(x)
    M, K = x.shape
    if out is None:
        out = _empty((1,), torch.float32, x.device)
    st = _lib.lib().bf16_amax(_ptr(x), M, K, ldx, _ptr(out), _stream(stream))
    _check(st, "bf16_amax")
    return out


def nvfp4_quantize_transpose(x, flags=ROWWISE | COLWISE, *, amax=None, global_scale=None,
                             q_row=None, s_row=None, q_t=None, s_t=None, workspace=None,
                             dev_err=None, stream=None):
    """bf16 x[M, K] -> NVFP4: q_row [M,K/2] / s_row [M,K/16] (ROWWISE),
    q_t [K,M/2] / s_t [K,M/16] (COLWISE), global_scale [1] fp32.  `amax`
    (1-element fp32 device tensor) skips the internal amax pass; flags | NVFP4_2D
    takes one scale per 16x16 block."""
    ldx = _input(x)
    M, K = x.shape
    dev = x.device
    out = {"global_scale": global_scale if global_scale is not None
           else _empty((1,), torch.float32, dev)}
    if flags & ROWWISE:
        out["q_row"] = q_row if q_row is not None else _empty((M, K // 2), torch.uint8, dev)
        out["s_row"] = s_row if s_row is not None else _empty((M, K // 16), torch.uint8, dev)
    if flags & COLWISE:
        out["q_t"] = q_t if q_t is not None else _empty((K, M // 2), torch.uint8, dev)
        out["s_t"] = s_t if s_t is not None else _empty((K, M // 16), torch.uint8, dev)
    ws_bytes = 0
    if amax is None:
        if workspace is None:
            workspace = _empty((16,), torch.uint8, dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.lib().nvfp4_quantize_transpose(
        _ptr(x), M, K, ldx, flags, _ptr(amax), _ptr(out["global_scale"]),
        _ptr(out.get("q_row")), _ptr(out.get("s_row")), _ptr(out.get("q_t")),
        _ptr(out.get("s_t")), _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream))
    _check(st, "nvfp4_quantize_transpose")
    return out


def mxq_selftest_bounded_wait(timeout_ns, dev_err, *, stream=None):
    """Run the bounded-wait self test (see include/mxq.h); the kernel sets
    DEVERR_TIMEOUT in dev_err (a 1-element int32 device tensor)."""
    st = _lib.lib().mxq_selftest_bounded_wait(int(timeout_ns), _ptr(dev_err), _stream(stream))
    _check(st, "mxq_selftest_bounded_wait")
