"""mx_quantize_rowcol_dbias_noalloc, the entry point for callers that cannot
allocate device memory (the library keeps its dbias scratch in a fixed device
array instead of a caller workspace).

Called through the C ABI and checked against mx_quantize_rowcol (which takes
a torch-allocated workspace) on two calls in a row with different shapes, so
contents left in the shared array by the first call cannot leak into the
second.  Codes and scales must match byte for byte; dbias within the dbias
tolerance of the other tests (1e-5 of sum |x| per column).  This file is
named to run last, so a failure here does not hide the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from parity_util import assert_equal_bytes, host, to_device

pytestmark = pytest.mark.gpu

mxq = pytest.importorskip("fp4_quantization_gb300")
from fp4_quantization_gb300 import _lib  # noqa: E402

BOTH = 3


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(x, flags):
    """Outputs allocated by the test, then one C-ABI call that allocates
    nothing; returns (status, outputs)."""
    M, K = x.shape
    dev = x.device
    out = {
        "q_row": torch.empty((M, K), dtype=torch.uint8, device=dev),
        "s_row": torch.empty((M, K // 32), dtype=torch.uint8, device=dev),
        "q_col": torch.empty((K, M), dtype=torch.uint8, device=dev),
        "s_col": torch.empty((K, M // 32), dtype=torch.uint8, device=dev),
        "dbias": torch.empty((K,), dtype=torch.float32, device=dev),
    }
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = _lib.lib().mx_quantize_rowcol_dbias_noalloc(
        _p(x), M, K, x.stride(0), flags, _p(out["q_row"]), _p(out["s_row"]), _p(out["q_col"]),
        _p(out["s_col"]), _p(out["dbias"]), _p(dev_err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    return st, out


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    for (M, K), seed in (((512, 768), 61), ((256, 1280), 62)):
        bits = synth.dbias(M=M, K=K, seed=seed)
        x = to_device(bits)
        ref = mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS)
        st, out = _noalloc(x, BOTH)
        assert st == 0, mxq.STATUS_NAMES.get(st, st)
        for key in ("q_row", "s_row", "q_col", "s_col"):
            assert_equal_bytes(host(out[key]), host(ref[key]), f"{M}x{K} {key}")
        tol = 1e-5 * np.abs(synth.bf16_bits_to_f32(bits).astype(np.float64)).sum(axis=0) + 1e-30
        err = np.abs(host(out["dbias"]).astype(np.float64) - host(ref["dbias"]).astype(np.float64))
        assert np.all(err <= tol), f"{M}x{K} dbias max err {err.max()}"


def test_noalloc_refuses_shapes_beyond_its_array():
    # ceil(32768 / 128) * 16384 * 4 bytes = 16 MiB of band sums > 8 MiB.
    L = _lib.lib()
    st = L.mx_quantize_rowcol_dbias_noalloc(None, 32768, 16384, 16384, BOTH, None, None, None,
                                            None, None, None, None)
    assert st == 5   # MXQ_EWORKSPACE
