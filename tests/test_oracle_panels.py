"""The row-panel runner the full-size GPU tests use: the oracle run panel
by panel on a thread pool assembles exactly the oracle's full-matrix output
(CPU only)."""
import numpy as np
import pytest

import oracle
import synth
from oracle_panels import mx_panels, nvfp4_panels, run_panels

BOTH = oracle.ROWWISE | oracle.COLWISE


def _same(a, b):
    assert sorted(a) == sorted(k for k in b if k in a)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("panel_rows", [32, 96, 160])
def test_mx_panels_equal_full_matrix(panel_rows):
    bits = synth.rowcol(M=320, K=192, seed=40)
    full = oracle.mx_quantize(bits, BOTH)
    got = run_panels(lambda r0, r1: oracle.mx_quantize(bits[r0:r1], BOTH), 320,
                     {"q_row": (0, 1), "s_row": (0, 1), "q_col": (1, 1), "s_col": (1, 1 / 32)},
                     panel_rows=panel_rows)
    _same(got, full)


def test_gated_and_backward_panels_equal_full_matrix():
    x = synth.swiglu(M=256, N=96, seed=41)
    grad = synth.gelu(M=256, K=96, seed=42)
    full = oracle.mx_quantize_gated(x, 96, act=oracle.ACT_GELU_TANH)
    _same(mx_panels(lambda r0, r1: oracle.mx_quantize_gated(x[r0:r1], 96,
                                                            act=oracle.ACT_GELU_TANH), 256), full)
    full = oracle.mx_quantize_dgated(grad, x, 96, oracle.ACT_SILU)
    _same(mx_panels(lambda r0, r1: oracle.mx_quantize_dgated(grad[r0:r1], x[r0:r1], 96,
                                                             oracle.ACT_SILU), 256), full)


@pytest.mark.parametrize("flags", [BOTH, BOTH | oracle.NVFP4_2D], ids=["1d", "2d"])
def test_nvfp4_panels_equal_full_matrix(flags):
    bits = synth.nvfp4(M=256, K=128, seed=43)
    A = oracle.bf16_amax(bits)
    full = oracle.nvfp4_quantize(bits, tensor_amax=A, flags=flags)
    got = nvfp4_panels(lambda r0, r1: oracle.nvfp4_quantize(bits[r0:r1], tensor_amax=A,
                                                            flags=flags), 256)
    _same(got, full)
