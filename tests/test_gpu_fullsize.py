"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (the same C-ABI calls on the same seeded inputs).

Every output is compared with the oracle over the WHOLE tensor: the oracle
runs in row panels on every host core (blocks never cross a panel, so the
panels give exactly the full-matrix output).  Plain casts, dbias codes and
NVFP4 are compared byte for byte; the fused-activation paths are counted
over the whole tensor against their budget (codes within one E4M3 step and
scales within one code, each in at most 1e-4 of the tensor), and the
measured fractions are reported (MXQ_PARITY_LOG collects them).  Only the
2^31-element shapes (4 GiB inputs) stay sampled in windows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle_panels import mx_panels, nvfp4_panels
from parity_util import (assert_activation_budget, assert_equal_bytes, count_activation_mismatches,
                         host, record, to_device)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import fp4_quantization_gb300 as mxq  # noqa: E402  (no skip: a missing libmxq.so is an error)

BOTH = 3


def windows(M, K, h, w, n, seed, align=32):
    """n random (m0, k0) windows of h x w (multiples of `align`) plus the
    four corners."""
    rng = np.random.default_rng(seed)
    out = [(0, 0), (M - h, 0), (0, K - w), (M - h, K - w)]
    for _ in range(n):
        out.append((int(rng.integers(0, (M - h) // align + 1)) * align,
                    int(rng.integers(0, (K - w) // align + 1)) * align))
    return out


def _exact(out, ref, what):
    for key in ref:
        assert_equal_bytes(host(out[key]), ref[key], f"{what} {key}")
    record(what, compared=sorted(ref), bytes=int(sum(ref[k].size for k in ref)), differ=0)


def _activation(out, ref, what, untile=None):
    """Whole-tensor counts of both directions against the budget."""
    for direction, qk, sk in (("row", "q_row", "s_row"), ("col", "q_col", "s_col")):
        if qk not in ref:
            continue
        s = host(out[sk])
        if untile is not None:
            s = untile(s, *ref[sk].shape)
        res = count_activation_mismatches(host(out[qk]), s, ref[qk], ref[sk])
        record(f"{what} {direction}", **res)
        assert_activation_budget(res, f"{what} {direction}")


def _dbias_check(got, ref, colsum_abs, what, rel):
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    tol = rel * colsum_abs + 1e-30
    ratio = err / (colsum_abs + 1e-30)
    record(what, max_err_over_sum_abs=float(ratio.max()), bound=rel,
           max_abs_err=float(err.max()))
    assert np.all(err <= tol), f"{what}: max err / tol {np.max(err / tol)}"


def test_rowcol_16384():
    bits = synth.rowcol()
    x = to_device(bits)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mxq.mx_quantize_rowcol(x, BOTH, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize(bits[r0:r1], BOTH), 16384)
    _exact(out, ref, "rowcol 16384x16384")
    # The scales again by their closed form over the whole output (bf16
    # exponent field of the block's largest magnitude - 8, floored at 0),
    # computed on the device from x alone.
    xb = x.view(torch.int16)
    mag = (xb & 0x7FFF).to(torch.int32)
    rmax = mag.view(16384, 512, 32).amax(dim=2)
    assert torch.equal(out["s_row"], torch.clamp((rmax >> 7) - 8, min=0).to(torch.uint8))
    cmax = mag.view(512, 32, 16384).amax(dim=1).t()
    assert torch.equal(out["s_col"], torch.clamp((cmax >> 7) - 8, min=0).to(torch.uint8))


def test_rowcol_8192x28672():
    bits = synth.rowcol(M=8192, K=28672)
    out = mxq.mx_quantize_rowcol(to_device(bits), BOTH)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize(bits[r0:r1], BOTH), 8192)
    _exact(out, ref, "rowcol 8192x28672")


def _untile(t, R, C):
    """Inverse of the 128 x 4 tiled scale layout (reshape form), cropped to
    [R, C]; the layout itself is pinned against the oracle at small sizes."""
    t = np.asarray(t)
    Rp, Cp = t.shape
    return t.reshape(Rp // 128, Cp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(Rp, Cp)[:R, :C]


def test_gemm_ready_rowcol_16384():
    """Ceil-style scale rule with scales in 128 x 4 tiles: codes byte for
    byte, scales byte for byte once untiled."""
    bits = synth.rowcol()
    out = mxq.mx_quantize_rowcol(to_device(bits), BOTH | mxq.SCALE_RCEIL | mxq.SCALE_SWIZZLED)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize(bits[r0:r1], BOTH | oracle.SCALE_RCEIL),
                    16384)
    for key in ("q_row", "q_col"):
        assert_equal_bytes(host(out[key]), ref[key], f"gemm-ready {key}")
    for key in ("s_row", "s_col"):
        assert_equal_bytes(_untile(host(out[key]), *ref[key].shape), ref[key], f"gemm-ready {key}")
    record("gemm-ready rowcol 16384x16384", differ=0)


def test_dim1_colwise_16384():
    bits = synth.dim1()
    out = mxq.mx_quantize_rowcol(to_device(bits), mxq.COLWISE)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize(bits[r0:r1], oracle.COLWISE), 16384)
    _exact(out, ref, "dim1 colwise 16384x16384")


def test_dbias_8192():
    bits = synth.dbias()
    out = mxq.mx_quantize_rowcol(to_device(bits), BOTH | mxq.DBIAS)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize(bits[r0:r1], BOTH), 8192)
    _exact({k: out[k] for k in ref}, ref, "dbias 8192x8192 codes")
    want = oracle.mx_quantize(bits, oracle.DBIAS)["dbias"]
    colsum = np.abs(synth.bf16_bits_to_f32(bits).astype(np.float64)).sum(axis=0)
    _dbias_check(host(out["dbias"]), want, colsum, "dbias 8192x8192", 1e-5)


def test_swiglu_8192x14336():
    bits = synth.swiglu()
    N = 14336
    out = mxq.mx_quantize_gated(to_device(bits), BOTH)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize_gated(bits[r0:r1], N, act=oracle.ACT_SILU),
                    8192)
    _activation(out, ref, "swiglu 8192x2x14336")


def test_geglu_8192x14336():
    bits = synth.swiglu()
    N = 14336
    out = mxq.mx_quantize_gated(to_device(bits), BOTH | mxq.ACT_GELU_TANH)
    ref = mx_panels(
        lambda r0, r1: oracle.mx_quantize_gated(bits[r0:r1], N, act=oracle.ACT_GELU_TANH), 8192)
    _activation(out, ref, "geglu 8192x2x14336")


def test_gelu_8192x14336():
    bits = synth.gelu()
    out = mxq.mx_quantize_rowcol(to_device(bits), BOTH | mxq.ACT_GELU_TANH)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize(bits[r0:r1], BOTH, act=oracle.ACT_GELU_TANH),
                    8192)
    _activation(out, ref, "gelu 8192x14336")


def test_dbias_dgelu_8192x14336():
    grad, xb = synth.gelu(seed=8), synth.gelu()
    out = mxq.mx_quantize_dact(to_device(grad), to_device(xb), BOTH | mxq.DBIAS | mxq.ACT_GELU_TANH)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize_dact(grad[r0:r1], xb[r0:r1],
                                                           oracle.ACT_GELU_TANH, BOTH), 8192)
    _activation(out, ref, "dbias_dgelu 8192x14336")
    want = oracle.mx_quantize_dact(grad, xb, oracle.ACT_GELU_TANH, oracle.DBIAS)["dbias"]
    # |gelu'| <= 1.2 bounds sum_m |y| by 1.2 sum_m |grad|.
    colsum = 1.2 * np.abs(synth.bf16_bits_to_f32(grad).astype(np.float64)).sum(axis=0)
    _dbias_check(host(out["dbias"]), want, colsum, "dbias_dgelu 8192x14336", 1e-5)


def test_dswiglu_8192x14336():
    grad, xb = synth.gelu(seed=9), synth.swiglu()
    N = 14336
    out = mxq.mx_quantize_dgated(to_device(grad), to_device(xb), BOTH)
    ref = mx_panels(lambda r0, r1: oracle.mx_quantize_dgated(grad[r0:r1], xb[r0:r1], N,
                                                             oracle.ACT_SILU), 8192)
    _activation(out, ref, "dswiglu 8192x14336")


@pytest.mark.parametrize("two_d", [False, True], ids=["1d", "2d"])
def test_nvfp4_16384x8192(two_d):
    bits = synth.nvfp4()
    flags = BOTH | (mxq.NVFP4_2D if two_d else 0)
    out = mxq.nvfp4_quantize_transpose(to_device(bits), flags)   # tensor amax on the device
    A = oracle.bf16_amax(bits)
    G = host(out["global_scale"])[0]
    assert G == np.float32(np.float32(A) / np.float32(2688.0))
    oflags = BOTH | (oracle.NVFP4_2D if two_d else 0)
    ref = nvfp4_panels(lambda r0, r1: oracle.nvfp4_quantize(bits[r0:r1], tensor_amax=A,
                                                            flags=oflags), 16384)
    _exact({k: out[k] for k in ref}, ref, f"nvfp4 {'2d' if two_d else '1d'} 16384x8192")


def _device_window(x, m0, k0, h, w):
    return x[m0:m0 + h, k0:k0 + w].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _edge_windows(M, K, h, w, n, seed, align):
    """Random windows plus the four corners (the last rows and columns are
    where a 32-bit index would have wrapped)."""
    return windows(M, K, h, w, n, seed, align) + [(0, 0), (0, K - w), (M - h, 0), (M - h, K - w)]


def test_rowcol_past_2e31_elements():
    """65536 x 32768 = 2^31 elements (4 GiB of bf16): element and byte
    offsets above 2^31 in every output."""
    M, K = 65536, 32768
    x = synth.device_normal(M, K, seed=76)
    out = mxq.mx_quantize_rowcol(x, BOTH)
    torch.cuda.synchronize()
    for m0, k0 in _edge_windows(M, K, 32, 256, 12, seed=8, align=32):
        bits = _device_window(x, m0, k0, 32, 256)
        ref = oracle.mx_quantize(bits, BOTH)
        assert_equal_bytes(host(out["q_row"][m0:m0 + 32, k0:k0 + 256]), ref["q_row"], f"q_row ({m0},{k0})")
        assert_equal_bytes(host(out["s_row"][m0:m0 + 32, k0 // 32:(k0 + 256) // 32]), ref["s_row"],
                           f"s_row ({m0},{k0})")
        assert_equal_bytes(host(out["q_col"][k0:k0 + 256, m0:m0 + 32]), ref["q_col"], f"q_col ({m0},{k0})")
        assert_equal_bytes(host(out["s_col"][k0:k0 + 256, m0 // 32:(m0 + 32) // 32]), ref["s_col"],
                           f"s_col ({m0},{k0})")
    del x, out
    torch.cuda.empty_cache()


def test_nvfp4_past_2e31_elements():
    """65536 x 32768 NVFP4 (1D), tensor amax computed on the device."""
    M, K = 65536, 32768
    x = synth.device_normal(M, K, seed=77)
    out = mxq.nvfp4_quantize_transpose(x, BOTH)
    A = float(host(mxq.bf16_amax(x))[0])
    assert A == float(x.abs().max().float().item())
    for m0, k0 in _edge_windows(M, K, 64, 128, 12, seed=9, align=16):
        bits = _device_window(x, m0, k0, 64, 128)
        ref = oracle.nvfp4_quantize(bits, tensor_amax=A)
        assert_equal_bytes(host(out["q_row"][m0:m0 + 64, k0 // 2:(k0 + 128) // 2]), ref["q_row"],
                           f"q_row ({m0},{k0})")
        assert_equal_bytes(host(out["s_row"][m0:m0 + 64, k0 // 16:(k0 + 128) // 16]), ref["s_row"],
                           f"s_row ({m0},{k0})")
        assert_equal_bytes(host(out["q_t"][k0:k0 + 128, m0 // 2:(m0 + 64) // 2]), ref["q_t"],
                           f"q_t ({m0},{k0})")
        assert_equal_bytes(host(out["s_t"][k0:k0 + 128, m0 // 16:(m0 + 64) // 16]), ref["s_t"],
                           f"s_t ({m0},{k0})")
    del x, out
    torch.cuda.empty_cache()
