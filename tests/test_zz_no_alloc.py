"""mx_quantize_rowcol_dbias_noalloc, the entry point for callers that cannot
allocate device memory (the library keeps its dbias scratch in a fixed device
array instead of a caller workspace).

Called through the C ABI and checked against mx_quantize_rowcol (which takes
a torch-allocated workspace): two calls in a row with different shapes, so
contents left in the shared array by the first call cannot leak into the
second; two calls queued back to back on one stream with no synchronisation
between them (the second call's band sums overwrite the array while the
first call's finalize may still be queued); and the largest shape the array
takes.  Codes and scales must match byte for byte; dbias within the dbias
tolerance of the other tests (1e-5 of sum |x| per column).  This file is
named to run last, so a failure here does not hide the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from parity_util import assert_equal_bytes, host, to_device

import fp4_quantization_gb300 as mxq  # noqa: E402  (no skip: a missing libmxq.so is an error)
from fp4_quantization_gb300 import _lib  # noqa: E402

BOTH = 3
ARRAY_BYTES = 8 << 20


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(M, K, dev):
    return {
        "q_row": torch.empty((M, K), dtype=torch.uint8, device=dev),
        "s_row": torch.empty((M, K // 32), dtype=torch.uint8, device=dev),
        "q_col": torch.empty((K, M), dtype=torch.uint8, device=dev),
        "s_col": torch.empty((K, M // 32), dtype=torch.uint8, device=dev),
        "dbias": torch.empty((K,), dtype=torch.float32, device=dev),
    }


def _enqueue_noalloc(x, flags, out, dev_err):
    """One C-ABI call that allocates nothing, on torch's current stream;
    returns the status without synchronising."""
    M, K = x.shape
    return _lib.lib().mx_quantize_rowcol_dbias_noalloc(
        _p(x), M, K, x.stride(0), flags, _p(out["q_row"]), _p(out["s_row"]), _p(out["q_col"]),
        _p(out["s_col"]), _p(out["dbias"]), _p(dev_err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _noalloc(x, flags):
    out = _outputs(*x.shape, x.device)
    dev_err = torch.zeros(1, dtype=torch.int32, device=x.device)
    st = _enqueue_noalloc(x, flags, out, dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    return st, out


def _check_against_allocating_path(bits, out, what):
    ref = mxq.mx_quantize_rowcol(to_device(bits), BOTH | mxq.DBIAS)
    for key in ("q_row", "s_row", "q_col", "s_col"):
        assert_equal_bytes(host(out[key]), host(ref[key]), f"{what} {key}")
    tol = 1e-5 * np.abs(synth.bf16_bits_to_f32(bits).astype(np.float64)).sum(axis=0) + 1e-30
    err = np.abs(host(out["dbias"]).astype(np.float64) - host(ref["dbias"]).astype(np.float64))
    assert np.all(err <= tol), f"{what} dbias max err {err.max()}"


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_on_two_calls():
    for (M, K), seed in (((512, 768), 61), ((256, 1280), 62)):
        bits = synth.dbias(M=M, K=K, seed=seed)
        st, out = _noalloc(to_device(bits), BOTH)
        assert st == 0, mxq.STATUS_NAMES.get(st, st)
        _check_against_allocating_path(bits, out, f"{M}x{K}")


@pytest.mark.gpu
def test_noalloc_two_calls_queued_without_synchronising():
    """Both calls on one stream, one synchronisation after the second: the
    second call's band sums must not reach the first call's dbias."""
    inputs = [synth.dbias(M=1024, K=2048, seed=seed) for seed in (63, 64)]
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xs = [to_device(bits) for bits in inputs]
    outs = [_outputs(1024, 2048, "cuda") for _ in inputs]
    torch.cuda.synchronize()
    for x, out in zip(xs, outs):
        assert _enqueue_noalloc(x, BOTH, out, dev_err) == 0
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    for i, (bits, out) in enumerate(zip(inputs, outs)):
        _check_against_allocating_path(bits, out, f"queued call {i}")


@pytest.mark.gpu
def test_noalloc_largest_shape_the_array_takes():
    """16384 x 16384 needs exactly the 8 MiB of the array: accepted, and the
    same bytes as the allocating entry point (compared on the device)."""
    M = K = 16384
    assert mxq.mxq_workspace_bytes(mxq.OP_ROWCOL, M, K, mxq.DBIAS) == ARRAY_BYTES
    x = synth.device_normal(M, K, seed=65)
    out = _outputs(M, K, x.device)
    dev_err = torch.zeros(1, dtype=torch.int32, device=x.device)
    assert _enqueue_noalloc(x, BOTH, out, dev_err) == 0
    ref = mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    for key in ("q_row", "s_row", "q_col", "s_col"):
        assert torch.equal(out[key], ref[key]), key
    tol = 1e-5 * x.float().abs().sum(dim=0).double() + 1e-30
    err = (out["dbias"].double() - ref["dbias"].double()).abs()
    assert bool((err <= tol).all()), f"dbias max err {err.max().item()}"
    del x, out, ref
    torch.cuda.empty_cache()


def test_noalloc_refuses_shapes_beyond_its_array():
    """Host-side: one band of 128 rows past 16384 x 16384 needs more than the
    array and is refused before anything is enqueued (no GPU needed)."""
    assert mxq.mxq_workspace_bytes(mxq.OP_ROWCOL, 16384 + 128, 16384, mxq.DBIAS) > ARRAY_BYTES
    L = _lib.lib()
    for M, K in ((16384 + 128, 16384), (32768, 16384), (16384, 16384 + 32)):
        st = L.mx_quantize_rowcol_dbias_noalloc(None, M, K, K, BOTH, None, None, None, None, None,
                                                None, None)
        assert st == 5, (M, K, st)   # MXQ_EWORKSPACE
