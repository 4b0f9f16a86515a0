"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (the same C-ABI calls on the same seeded inputs).  The oracle
checks sampled windows -- every block is independent, so a window of x gives
exactly the blocks of the full output it covers -- plus the last rows and
columns, and whole-tensor properties where they are cheap (the tensor amax,
every dbias column)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import assert_equal_bytes, check_activation_blocks, host, to_device

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


def check_mx_windows(bits, out, flags, wins, h=32, w=256, act=oracle.ACT_NONE, exact=True):
    for m0, k0 in wins:
        ref = oracle.mx_quantize(bits[m0:m0 + h, k0:k0 + w], flags, act=act)
        got = {}
        if flags & oracle.ROWWISE:
            got["q_row"] = host(out["q_row"][m0:m0 + h, k0:k0 + w])
            got["s_row"] = host(out["s_row"][m0:m0 + h, k0 // 32:(k0 + w) // 32])
        if flags & oracle.COLWISE:
            got["q_col"] = host(out["q_col"][k0:k0 + w, m0:m0 + h])
            got["s_col"] = host(out["s_col"][k0:k0 + w, m0 // 32:(m0 + h) // 32])
        if exact:
            for key in got:
                assert_equal_bytes(got[key], ref[key], f"window ({m0},{k0}) {key}")
        else:
            if "q_row" in got:
                check_activation_blocks(got["q_row"], got["s_row"], ref["q_row"], ref["s_row"], 1,
                                        f"window ({m0},{k0}) row")
            if "q_col" in got:
                check_activation_blocks(got["q_col"], got["s_col"], ref["q_col"], ref["s_col"], 1,
                                        f"window ({m0},{k0}) col")


def test_rowcol_16384():
    bits = synth.rowcol()
    x = to_device(bits)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mxq.mx_quantize_rowcol(x, BOTH, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    check_mx_windows(bits, out, BOTH, windows(16384, 16384, 32, 256, 60, seed=1))
    # Property over the whole output: every scale is the closed form of its
    # block's largest magnitude (bf16 exponent field - 8, floored at 0).
    xb = x.view(torch.int16)
    mag = (xb & 0x7FFF).to(torch.int32)
    rmax = mag.view(16384, 512, 32).amax(dim=2)
    want = torch.clamp((rmax >> 7) - 8, min=0).to(torch.uint8)
    assert torch.equal(out["s_row"], want)
    cmax = mag.view(512, 32, 16384).amax(dim=1).t()
    want = torch.clamp((cmax >> 7) - 8, min=0).to(torch.uint8)
    assert torch.equal(out["s_col"], want)


def test_dim1_colwise_16384():
    bits = synth.dim1()
    x = to_device(bits)
    out = mxq.mx_quantize_rowcol(x, mxq.COLWISE)
    check_mx_windows(bits, out, oracle.COLWISE, windows(16384, 16384, 32, 256, 60, seed=2))


def test_dbias_8192():
    bits = synth.dbias()
    x = to_device(bits)
    out = mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS)
    check_mx_windows(bits, out, BOTH, windows(8192, 8192, 32, 256, 40, seed=3))
    ref = oracle.mx_quantize(bits, oracle.DBIAS)["dbias"].astype(np.float64)
    got = host(out["dbias"]).astype(np.float64)
    tol = 1e-5 * np.abs(synth.bf16_bits_to_f32(bits).astype(np.float64)).sum(axis=0) + 1e-30
    assert np.all(np.abs(got - ref) <= tol), f"max err / tol {np.max(np.abs(got - ref) / tol)}"


def test_swiglu_8192x14336():
    bits = synth.swiglu()
    x = to_device(bits)
    out = mxq.mx_quantize_gated(x, BOTH)
    N = 14336
    for m0, k0 in windows(8192, N, 32, 256, 40, seed=4):
        sub = np.ascontiguousarray(np.concatenate([bits[m0:m0 + 32, k0:k0 + 256],
                                                   bits[m0:m0 + 32, N + k0:N + k0 + 256]], axis=1))
        ref = oracle.mx_quantize_swiglu(sub, 256)
        check_activation_blocks(host(out["q_row"][m0:m0 + 32, k0:k0 + 256]),
                                host(out["s_row"][m0:m0 + 32, k0 // 32:k0 // 32 + 8]),
                                ref["q_row"], ref["s_row"], 1, f"swiglu row ({m0},{k0})")
        check_activation_blocks(host(out["q_col"][k0:k0 + 256, m0:m0 + 32]),
                                host(out["s_col"][k0:k0 + 256, m0 // 32:m0 // 32 + 1]),
                                ref["q_col"], ref["s_col"], 1, f"swiglu col ({m0},{k0})")


def test_gelu_8192x14336():
    bits = synth.gelu()
    x = to_device(bits)
    out = mxq.mx_quantize_rowcol(x, BOTH | mxq.ACT_GELU_TANH)
    check_mx_windows(bits, out, BOTH, windows(8192, 14336, 32, 256, 40, seed=5),
                     act=oracle.ACT_GELU_TANH, exact=False)


def test_nvfp4_16384x8192():
    bits = synth.nvfp4()
    x = to_device(bits)
    out = mxq.nvfp4_quantize_transpose(x, BOTH)
    A = oracle.bf16_amax(bits)
    G = host(out["global_scale"])[0]
    assert G == np.float32(np.float32(A) / np.float32(2688.0))
    for m0, k0 in windows(16384, 8192, 64, 128, 50, seed=6, align=16):
        ref = oracle.nvfp4_quantize(bits[m0:m0 + 64, k0:k0 + 128], tensor_amax=A)
        assert_equal_bytes(host(out["q_row"][m0:m0 + 64, k0 // 2:(k0 + 128) // 2]), ref["q_row"],
                           f"nvfp4 q_row ({m0},{k0})")
        assert_equal_bytes(host(out["s_row"][m0:m0 + 64, k0 // 16:(k0 + 128) // 16]), ref["s_row"],
                           f"nvfp4 s_row ({m0},{k0})")
        assert_equal_bytes(host(out["q_t"][k0:k0 + 128, m0 // 2:(m0 + 64) // 2]), ref["q_t"],
                           f"nvfp4 q_t ({m0},{k0})")
        assert_equal_bytes(host(out["s_t"][k0:k0 + 128, m0 // 16:(m0 + 64) // 16]), ref["s_t"],
                           f"nvfp4 s_t ({m0},{k0})")


def test_nvfp4_2d_16384x8192():
    """16x16 blocks at the NVFP4 workload size, windows aligned to blocks."""
    bits = synth.nvfp4()
    x = to_device(bits)
    out = mxq.nvfp4_quantize_transpose(x, BOTH | mxq.NVFP4_2D)
    A = oracle.bf16_amax(bits)
    for m0, k0 in windows(16384, 8192, 64, 128, 40, seed=7, align=16):
        ref = oracle.nvfp4_quantize(bits[m0:m0 + 64, k0:k0 + 128], tensor_amax=A,
                                    flags=BOTH | oracle.NVFP4_2D)
        assert_equal_bytes(host(out["q_row"][m0:m0 + 64, k0 // 2:(k0 + 128) // 2]), ref["q_row"],
                           f"2d q_row ({m0},{k0})")
        assert_equal_bytes(host(out["s_row"][m0:m0 + 64, k0 // 16:(k0 + 128) // 16]), ref["s_row"],
                           f"2d s_row ({m0},{k0})")
        assert_equal_bytes(host(out["q_t"][k0:k0 + 128, m0 // 2:(m0 + 64) // 2]), ref["q_t"],
                           f"2d q_t ({m0},{k0})")
        assert_equal_bytes(host(out["s_t"][k0:k0 + 128, m0 // 16:(m0 + 64) // 16]), ref["s_t"],
                           f"2d s_t ({m0},{k0})")


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
