"""GPU parity: the CUDA path through the C ABI against the oracle, element
by element, on seeded inputs that span several tiles and a ragged tail.

Bars: plain casts, dbias codes and NVFP4 bit-exact; dbias within 1e-5 of
sum|x| per column; GELU / SwiGLU codes within one E4M3 step in at most 1e-4
of the elements (and scales within one code in at most 1e-4 of the blocks).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (assert_equal_bytes, check_activation_blocks, host, to_device)

pytestmark = pytest.mark.gpu

import fp4_quantization_gb300 as mxq  # noqa: E402  (no skip: a missing libmxq.so is an error)

BOTH = 3


def _rowcol_cases():
    return [
        ("plain_small", synth.plain_small(), 0),
        ("multi_tile_ragged_k", synth.dbias(M=96, K=352, seed=31), 0),
        ("tall_thin", synth.rowcol(M=640, K=32, seed=32), 0),
        ("wide_short", synth.dim1(M=32, K=1056, seed=33), 0),
        ("many_tiles", synth.dbias(M=512, K=1024, seed=34), 0),
        # colwise scale rows of 5 bytes (M / 32 = 5: unaligned 4-byte runs)
        # and a last band of 32 rows
        ("odd_scale_rows", synth.rowcol(M=160, K=288, seed=35), 0),
        # 33 bands, the last one 32 rows, over 2 tiles along K
        ("ragged_last_band", synth.rowcol(M=4128, K=160, seed=36), 0),
    ]


@pytest.mark.parametrize("name,bits,_", _rowcol_cases(), ids=[c[0] for c in _rowcol_cases()])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_mx_rowcol_bit_exact(name, bits, _, flags):
    x = to_device(bits)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mxq.mx_quantize_rowcol(x, flags, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    ref = oracle.mx_quantize(bits, flags)
    for key in ref:
        assert_equal_bytes(host(out[key]), ref[key], f"{name} {key}")


@pytest.mark.parametrize("M,K,seed", [(3104, 2080, 48), (8192, 4096, 49), (16384, 1280, 60)],
                         ids=["ragged_groups", "whole_groups", "scale_rows_8_aligned"])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_mx_rowcol_cta_ranges(M, K, seed, flags):
    """Enough 128x128 steps that every SM walks a range of them: the first
    shape has a ragged last band group and ragged K, with CTA ranges of two
    or three steps that start and end inside band groups; the second gives
    each CTA about thirteen steps, so some ranges cover whole groups and
    their scale bytes leave in full runs; the third has rowwise scale rows of
    40 bytes (8- but not 16-byte aligned), whose full 8-step runs must not
    take the 16-byte store path."""
    bits = synth.rowcol(M=M, K=K, seed=seed)
    x = to_device(bits)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mxq.mx_quantize_rowcol(x, flags, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    ref = oracle.mx_quantize(bits, flags)
    for key in ref:
        assert_equal_bytes(host(out[key]), ref[key], f"{M}x{K} {key}")


@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("M", [4192, 4224, 8288], ids=["m4192", "m4224", "m8288"])
def test_mx_rowcol_host_buffers(flags, pinned, M):
    """The host-buffer entry point: three row panels (2048, 2048 and 96 or
    128 rows; the whole-matrix colwise scale rows are 131 bytes, written byte
    by byte, or 132, written by 4-byte runs) or five (4 x 2048 + 96), ragged
    K, outputs equal to the device path's byte for byte."""
    bits = synth.rowcol(M=M, K=1056, seed=74)
    x_host = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    if pinned:
        x_host = x_host.pin_memory()
    out = mxq.mx_quantize_rowcol_host(x_host, flags)
    torch.cuda.synchronize()
    ref = mxq.mx_quantize_rowcol(to_device(bits), flags)
    for key in ref:
        assert_equal_bytes(out[key].numpy(), host(ref[key]), f"host path {key}")


def test_mx_rowcol_host_strided_window():
    """ldx > K: a column window of a wider host matrix, one panel."""
    full = synth.rowcol(M=256, K=640, seed=75)
    x_host = torch.from_numpy(full.view(np.int16)).view(torch.bfloat16)[:, 64:64 + 512]
    out = mxq.mx_quantize_rowcol_host(x_host, BOTH)
    torch.cuda.synchronize()
    ref = oracle.mx_quantize(full[:, 64:64 + 512], BOTH)
    for key in ref:
        assert_equal_bytes(out[key].numpy(), ref[key], f"host window {key}")


@pytest.mark.parametrize("name,bits", [("plain_small", synth.plain_small()),
                                       ("dbias_blocks", synth.dbias(M=512, K=1024, seed=79)),
                                       ("ragged", synth.rowcol(M=3104, K=2080, seed=80))],
                         ids=["plain_small", "dbias_blocks", "ragged"])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_mx_rowcol_rceil(name, bits, flags):
    """Ceil-style scale rule: bit-exact, including zero, subnormal and
    outlier blocks."""
    out = mxq.mx_quantize_rowcol(to_device(bits), flags | mxq.SCALE_RCEIL)
    ref = oracle.mx_quantize(bits, flags | oracle.SCALE_RCEIL)
    for key in ref:
        assert_equal_bytes(host(out[key]), ref[key], f"rceil {name} {key}")


def test_mx_rceil_fused_paths():
    """The ceil rule on dbias (exact codes), GELU, SwiGLU and dGELU
    (activation tolerance), and the host-buffer path."""
    bits = synth.dbias(M=320, K=224, seed=81)
    out = mxq.mx_quantize_rowcol(to_device(bits), BOTH | mxq.DBIAS | mxq.SCALE_RCEIL)
    ref = oracle.mx_quantize(bits, BOTH | oracle.DBIAS | oracle.SCALE_RCEIL)
    for key in ("q_row", "s_row", "q_col", "s_col"):
        assert_equal_bytes(host(out[key]), ref[key], f"rceil dbias {key}")
    g = synth.gelu(M=256, K=384, seed=82)
    out = mxq.mx_quantize_rowcol(to_device(g), BOTH | mxq.ACT_GELU_TANH | mxq.SCALE_RCEIL)
    _check_mx_tol(out, oracle.mx_quantize(g, BOTH | oracle.SCALE_RCEIL, act=oracle.ACT_GELU_TANH),
                  "rceil gelu")
    sw = synth.swiglu(M=256, N=352, seed=83)
    out = mxq.mx_quantize_gated(to_device(sw), BOTH | mxq.SCALE_RCEIL)
    _check_mx_tol(out, oracle.mx_quantize_gated(sw, 352, flags=BOTH | oracle.SCALE_RCEIL),
                  "rceil swiglu")
    gr = synth.gelu(M=256, K=384, seed=84)
    out = mxq.mx_quantize_dact(to_device(gr), to_device(g), BOTH | mxq.ACT_GELU_TANH | mxq.SCALE_RCEIL)
    _check_mx_tol(out, oracle.mx_quantize_dact(gr, g, oracle.ACT_GELU_TANH, BOTH | oracle.SCALE_RCEIL),
                  "rceil dgelu")
    hb = synth.rowcol(M=2176, K=320, seed=85)
    xh = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16).pin_memory()
    out = mxq.mx_quantize_rowcol_host(xh, BOTH | mxq.SCALE_RCEIL)
    torch.cuda.synchronize()
    ref = oracle.mx_quantize(hb, BOTH | oracle.SCALE_RCEIL)
    for key in ref:
        assert_equal_bytes(out[key].numpy(), ref[key], f"rceil host {key}")


def _untile(t, R, C):
    """Inverse of the 128 x 4 tiled scale layout (reshape form), cropped to
    [R, C]."""
    t = np.asarray(t)
    Rp, Cp = t.shape
    return t.reshape(Rp // 128, Cp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(Rp, Cp)[:R, :C]


@pytest.mark.parametrize("name,bits", [("plain_small", synth.plain_small()),
                                       ("ragged", synth.rowcol(M=3104, K=2080, seed=86)),
                                       ("whole_groups", synth.dim1(M=8192, K=1024, seed=87))],
                         ids=["plain_small", "ragged", "whole_groups"])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_mx_rowcol_tiled_scales(name, bits, flags):
    """Scales in the 128 x 4 tiled layout, padding included, byte for byte."""
    out = mxq.mx_quantize_rowcol(to_device(bits), flags | mxq.SCALE_SWIZZLED)
    ref = oracle.mx_quantize(bits, flags | oracle.SCALE_SWIZZLED)
    for key in ref:
        assert_equal_bytes(host(out[key]), ref[key], f"tiled {name} {key}")


def test_mx_tiled_scales_fused_paths():
    bits = synth.dbias(M=320, K=224, seed=88)
    out = mxq.mx_quantize_rowcol(to_device(bits), BOTH | mxq.DBIAS | mxq.SCALE_SWIZZLED)
    ref = oracle.mx_quantize(bits, BOTH | oracle.DBIAS | oracle.SCALE_SWIZZLED)
    for key in ("q_row", "s_row", "q_col", "s_col"):
        assert_equal_bytes(host(out[key]), ref[key], f"tiled dbias {key}")
    g = synth.gelu(M=256, K=384, seed=89)
    out = mxq.mx_quantize_rowcol(to_device(g), BOTH | mxq.ACT_GELU_TANH | mxq.SCALE_SWIZZLED)
    ref = oracle.mx_quantize(g, BOTH, act=oracle.ACT_GELU_TANH)
    check_activation_blocks(host(out["q_row"]), _untile(host(out["s_row"]), 256, 12), ref["q_row"],
                            ref["s_row"], 1, "tiled gelu row")
    check_activation_blocks(host(out["q_col"]), _untile(host(out["s_col"]), 384, 8), ref["q_col"],
                            ref["s_col"], 1, "tiled gelu col")
    x = synth.swiglu(M=256, N=256, seed=90)
    grad = synth.gelu(M=256, K=256, seed=91)
    out = mxq.mx_quantize_dgated(to_device(grad), to_device(x), BOTH | mxq.SCALE_SWIZZLED)
    ref = oracle.mx_quantize_dgated(grad, x, 256, oracle.ACT_SILU)
    check_activation_blocks(host(out["q_row"]), _untile(host(out["s_row"]), 256, 16), ref["q_row"],
                            ref["s_row"], 1, "tiled dswiglu row")
    check_activation_blocks(host(out["q_col"]), _untile(host(out["s_col"]), 512, 8), ref["q_col"],
                            ref["s_col"], 1, "tiled dswiglu col")
    with pytest.raises(mxq.MxqError):
        mxq.mx_quantize_dgated(to_device(synth.gelu(M=64, K=96, seed=92)),
                               to_device(synth.swiglu(M=64, N=96, seed=93)), BOTH | mxq.SCALE_SWIZZLED)
    for M in (4192, 8288):   # three and five row panels
        hb = synth.rowcol(M=M, K=1056, seed=94)
        xh = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16).pin_memory()
        out = mxq.mx_quantize_rowcol_host(xh, BOTH | mxq.SCALE_SWIZZLED)
        torch.cuda.synchronize()
        ref = oracle.mx_quantize(hb, BOTH | oracle.SCALE_SWIZZLED)
        for key in ref:
            assert_equal_bytes(out[key].numpy(), ref[key], f"tiled host M={M} {key}")


def test_mx_rowcol_strided_input():
    """ldx > K: a column window of a wider matrix."""
    full = synth.rowcol(M=128, K=512, seed=35)
    x = to_device(full)[:, 64:64 + 320]
    out = mxq.mx_quantize_rowcol(x, BOTH)
    ref = oracle.mx_quantize(full[:, 64:64 + 320], BOTH)
    for key in ref:
        assert_equal_bytes(host(out[key]), ref[key], key)


def test_mx_rowcol_repeat_is_deterministic():
    bits = synth.dbias(M=256, K=384, seed=36)
    x = to_device(bits)
    a = mxq.mx_quantize_rowcol(x, BOTH)
    b = mxq.mx_quantize_rowcol(x, BOTH)
    for key in a:
        assert torch.equal(a[key], b[key])


def _dbias_tolerance(bits):
    xv = synth.bf16_bits_to_f32(bits).astype(np.float64)
    return 1e-5 * np.abs(xv).sum(axis=0) + 1e-30


@pytest.mark.parametrize("M,K,seed", [(320, 224, 37), (32, 96, 38), (1024, 640, 39),
                                      (3104, 2080, 50)])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_mx_dbias(M, K, seed, flags):
    """Every direction: the column sums are taken in whichever pass widens
    the values (the colwise one, else the rowwise one)."""
    bits = synth.dbias(M=M, K=K, seed=seed)
    x = to_device(bits)
    out = mxq.mx_quantize_rowcol(x, flags | mxq.DBIAS)
    ref = oracle.mx_quantize(bits, flags | oracle.DBIAS)
    for key in ("q_row", "s_row", "q_col", "s_col"):
        if key in ref:
            assert_equal_bytes(host(out[key]), ref[key], f"dbias {key}")
    err = np.abs(host(out["dbias"]).astype(np.float64) - ref["dbias"].astype(np.float64))
    assert np.all(err <= _dbias_tolerance(bits)), f"dbias max err {err.max()}"


def test_mx_dbias_is_deterministic():
    """The column sums are added in a fixed order: repeated calls give the
    same bits."""
    x = to_device(synth.dbias(M=3104, K=2080, seed=50))
    a = mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS)
    b = mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS)
    assert torch.equal(a["dbias"], b["dbias"])


@pytest.mark.parametrize("M,K,seed", [(256, 384, 40), (2080, 1184, 51)])
def test_mx_gelu(M, K, seed):
    bits = synth.gelu(M=M, K=K, seed=seed)
    x = to_device(bits)
    out = mxq.mx_quantize_rowcol(x, BOTH | mxq.ACT_GELU_TANH)
    ref = oracle.mx_quantize(bits, BOTH, act=oracle.ACT_GELU_TANH)
    check_activation_blocks(host(out["q_row"]), host(out["s_row"]), ref["q_row"], ref["s_row"], 1, "gelu row")
    check_activation_blocks(host(out["q_col"]), host(out["s_col"]), ref["q_col"], ref["s_col"], 1, "gelu col")


@pytest.mark.parametrize("M,N,seed", [(256, 352, 41), (64, 128, 42), (2080, 1184, 52)])
def test_mx_swiglu(M, N, seed):
    bits = synth.swiglu(M=M, N=N, seed=seed)
    x = to_device(bits)
    out = mxq.mx_quantize_gated(x, BOTH)
    ref = oracle.mx_quantize_swiglu(bits, N)
    check_activation_blocks(host(out["q_row"]), host(out["s_row"]), ref["q_row"], ref["s_row"], 1, "swiglu row")
    check_activation_blocks(host(out["q_col"]), host(out["s_col"]), ref["q_col"], ref["s_col"], 1, "swiglu col")


def test_mx_swiglu_row_only_and_col_only():
    bits = synth.swiglu(M=96, N=160, seed=43)
    x = to_device(bits)
    ref = oracle.mx_quantize_swiglu(bits, 160)
    r = mxq.mx_quantize_gated(x, mxq.ROWWISE)
    c = mxq.mx_quantize_gated(x, mxq.COLWISE)
    check_activation_blocks(host(r["q_row"]), host(r["s_row"]), ref["q_row"], ref["s_row"], 1, "row")
    check_activation_blocks(host(c["q_col"]), host(c["s_col"]), ref["q_col"], ref["s_col"], 1, "col")


def _check_mx_tol(out, ref, what):
    for d in ("row", "col"):
        if f"q_{d}" in ref:
            check_activation_blocks(host(out[f"q_{d}"]), host(out[f"s_{d}"]), ref[f"q_{d}"],
                                    ref[f"s_{d}"], 1, f"{what} {d}")


@pytest.mark.parametrize("M,N,seed", [(256, 352, 62), (2080, 1184, 63)])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_mx_geglu(M, N, seed, flags):
    bits = synth.swiglu(M=M, N=N, seed=seed)
    out = mxq.mx_quantize_gated(to_device(bits), flags | mxq.ACT_GELU_TANH)
    ref = oracle.mx_quantize_gated(bits, N, act=oracle.ACT_GELU_TANH, flags=flags)
    _check_mx_tol(out, ref, "geglu")


@pytest.mark.parametrize("act", ["gelu", "silu"])
@pytest.mark.parametrize("M,K,seed,flags", [(320, 224, 64, BOTH), (2080, 1184, 65, BOTH),
                                            (2080, 1184, 66, mxq.ROWWISE),
                                            (2080, 1184, 67, mxq.COLWISE)])
def test_mx_dact(act, M, K, seed, flags):
    """grad * act'(x): both inputs N(0,1) (grad from the GELU recipe with
    another seed)."""
    x = synth.gelu(M=M, K=K, seed=seed)
    grad = synth.gelu(M=M, K=K, seed=seed + 100)
    f_gpu = mxq.ACT_GELU_TANH if act == "gelu" else mxq.ACT_SILU
    f_orc = oracle.ACT_GELU_TANH if act == "gelu" else oracle.ACT_SILU
    out = mxq.mx_quantize_dact(to_device(grad), to_device(x), flags | f_gpu)
    ref = oracle.mx_quantize_dact(grad, x, f_orc, flags)
    _check_mx_tol(out, ref, f"d{act}")


@pytest.mark.parametrize("act", ["gelu", "silu"])
@pytest.mark.parametrize("M,K,seed", [(320, 224, 68), (2080, 1184, 69)])
def test_mx_dbias_dact(act, M, K, seed):
    """dbias of y = grad * act'(x): |act'| <= 1.2 for both activations, so
    1e-5 * 1.2 * sum|grad| bounds 1e-5 * sum|y| per column."""
    x = synth.dbias(M=M, K=K, seed=seed)
    grad = synth.gelu(M=M, K=K, seed=seed + 100)
    f_gpu = mxq.ACT_GELU_TANH if act == "gelu" else mxq.ACT_SILU
    f_orc = oracle.ACT_GELU_TANH if act == "gelu" else oracle.ACT_SILU
    out = mxq.mx_quantize_dact(to_device(grad), to_device(x), BOTH | mxq.DBIAS | f_gpu)
    ref = oracle.mx_quantize_dact(grad, x, f_orc, BOTH | oracle.DBIAS)
    _check_mx_tol(out, ref, f"dbias_d{act}")
    tol = 1.2e-5 * np.abs(synth.bf16_bits_to_f32(grad).astype(np.float64)).sum(axis=0) + 1e-30
    err = np.abs(host(out["dbias"]).astype(np.float64) - ref["dbias"].astype(np.float64))
    assert np.all(err <= tol), f"dbias max err {err.max()}"


@pytest.mark.parametrize("act", ["silu", "gelu"])
@pytest.mark.parametrize("M,N,seed,flags", [(256, 352, 70, BOTH), (2080, 1184, 71, BOTH),
                                            (2080, 1184, 72, mxq.ROWWISE),
                                            (2080, 1184, 73, mxq.COLWISE)])
def test_mx_dgated(act, M, N, seed, flags):
    """[grad * up * act'(gate) | grad * act(gate)]; N = 352 and 1184 leave a
    ragged last 128-column tile in each half."""
    x = synth.swiglu(M=M, N=N, seed=seed)
    grad = synth.gelu(M=M, K=N, seed=seed + 100)
    f_gpu = mxq.ACT_GELU_TANH if act == "gelu" else mxq.ACT_SILU
    f_orc = oracle.ACT_GELU_TANH if act == "gelu" else oracle.ACT_SILU
    out = mxq.mx_quantize_dgated(to_device(grad), to_device(x), flags | f_gpu)
    ref = oracle.mx_quantize_dgated(grad, x, N, f_orc, flags=flags)
    _check_mx_tol(out, ref, f"d{act}glu")


@pytest.mark.parametrize("M,K,seed", [(224, 160, 44), (32, 32, 45), (64, 64, 46), (512, 320, 47),
                                      (768, 1600, 48), (32768, 640, 61)])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_nvfp4_bit_exact(M, K, seed, flags):
    bits = synth.nvfp4(M=M, K=K, seed=seed)
    x = to_device(bits)
    out = mxq.nvfp4_quantize_transpose(x, flags)
    ref = oracle.nvfp4_quantize(bits, flags=flags)
    assert host(out["global_scale"])[0] == np.float32(ref["global_scale"])
    for key in ("q_row", "s_row", "q_t", "s_t"):
        if key in ref:
            assert_equal_bytes(host(out[key]), ref[key], f"nvfp4 {key}")


def test_nvfp4_given_amax_and_hand_block():
    """A caller-supplied amax of 2688 makes the global scale exactly 1."""
    f = np.zeros((32, 32), np.float32)
    f[0, :12] = [6, 3, -1.5, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.0, 1]
    bits = synth.f32_to_bf16_bits(f)
    x = to_device(bits)
    amax = torch.tensor([2688.0], dtype=torch.float32, device="cuda")
    out = mxq.nvfp4_quantize_transpose(x, BOTH, amax=amax)
    ref = oracle.nvfp4_quantize(bits, tensor_amax=2688.0)
    assert host(out["global_scale"])[0] == 1.0
    for key in ("q_row", "s_row", "q_t", "s_t"):
        assert_equal_bytes(host(out[key]), ref[key], key)
    assert host(out["s_row"])[0, 0] == 0x38


@pytest.mark.parametrize("amax_factor", [0.25, 1.0, 3.0])
def test_nvfp4_caller_amax(amax_factor):
    """A caller amax below the data's (block amaxes beyond its binade take the
    saturated scale, code 0x7E), equal to it, and above it."""
    bits = synth.nvfp4(M=256, K=512, seed=51)
    A = np.float32(oracle.bf16_amax(bits) * amax_factor)
    x = to_device(bits)
    out = mxq.nvfp4_quantize_transpose(x, BOTH, amax=torch.tensor([A], device="cuda"))
    ref = oracle.nvfp4_quantize(bits, tensor_amax=float(A))
    assert host(out["global_scale"])[0] == np.float32(ref["global_scale"])
    for key in ("q_row", "s_row", "q_t", "s_t"):
        assert_equal_bytes(host(out[key]), ref[key], f"amax x{amax_factor} {key}")


def test_nvfp4_wide_dynamic_range():
    """Zero blocks, bf16 subnormal blocks and x1000 outliers: magnitudes far
    below the scale table's 21 binades must still get code 0."""
    bits = synth.dbias(M=512, K=256, seed=52)
    x = to_device(bits)
    out = mxq.nvfp4_quantize_transpose(x, BOTH)
    ref = oracle.nvfp4_quantize(bits)
    for key in ("q_row", "s_row", "q_t", "s_t"):
        assert_equal_bytes(host(out[key]), ref[key], f"wide range {key}")


def test_nvfp4_zero_tensor():
    bits = np.zeros((64, 64), np.uint16)
    bits[3, 5] = 0x8000
    out = mxq.nvfp4_quantize_transpose(to_device(bits), BOTH)
    ref = oracle.nvfp4_quantize(bits)
    assert host(out["global_scale"])[0] == 0.0
    for key in ("q_row", "s_row", "q_t", "s_t"):
        assert_equal_bytes(host(out[key]), ref[key], key)


@pytest.mark.parametrize("M,K,seed", [(224, 160, 53), (32, 32, 54), (512, 320, 55),
                                      (768, 1600, 56), (3104, 2080, 57), (32768, 640, 59)])
@pytest.mark.parametrize("flags", [BOTH, mxq.ROWWISE, mxq.COLWISE], ids=["both", "row", "col"])
def test_nvfp4_2d_bit_exact(M, K, seed, flags):
    """16x16 blocks: several CTA steps, ragged bands and ranges."""
    bits = synth.nvfp4(M=M, K=K, seed=seed)
    x = to_device(bits)
    out = mxq.nvfp4_quantize_transpose(x, flags | mxq.NVFP4_2D)
    ref = oracle.nvfp4_quantize(bits, flags=flags | oracle.NVFP4_2D)
    assert host(out["global_scale"])[0] == np.float32(ref["global_scale"])
    for key in ("q_row", "s_row", "q_t", "s_t"):
        if key in ref:
            assert_equal_bytes(host(out[key]), ref[key], f"nvfp4 2d {key}")


@pytest.mark.parametrize("amax_factor", [0.25, 1.0, 3.0])
def test_nvfp4_2d_caller_amax_and_wide_range(amax_factor):
    """Caller amax below, at and above the data's, on an input with zero and
    subnormal blocks and outliers."""
    bits = synth.dbias(M=256, K=512, seed=58)
    A = np.float32(oracle.bf16_amax(bits) * amax_factor)
    x = to_device(bits)
    out = mxq.nvfp4_quantize_transpose(x, BOTH | mxq.NVFP4_2D,
                                       amax=torch.tensor([A], device="cuda"))
    ref = oracle.nvfp4_quantize(bits, tensor_amax=float(A), flags=BOTH | oracle.NVFP4_2D)
    for key in ("q_row", "s_row", "q_t", "s_t"):
        assert_equal_bytes(host(out[key]), ref[key], f"2d amax x{amax_factor} {key}")


def _scaled_bits(bits, factor):
    return synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(bits) * np.float32(factor))


def _nvfp4_case(bits, A, flags, what):
    x = to_device(bits)
    amax = None if A is None else torch.tensor([np.float32(A)], device="cuda")
    out = mxq.nvfp4_quantize_transpose(x, flags, amax=amax)
    ref = oracle.nvfp4_quantize(bits, flags=flags,
                                **({} if A is None else {"tensor_amax": float(np.float32(A))}))
    assert host(out["global_scale"])[0] == np.float32(ref["global_scale"]), what
    for key in ("q_row", "s_row", "q_t", "s_t"):
        assert_equal_bytes(host(out[key]), ref[key], f"{what} {key}")


@pytest.mark.parametrize("two_d", [False, True], ids=["1d", "2d"])
def test_nvfp4_exact_ties(two_d):
    """G = 1 (caller amax 2688) and values 6 * (j / 16) * 2^e with j in
    16..31: for odd j the block's (b / 6) / G is exactly halfway between two
    E4M3 values, the case a one-multiply estimate of the quotient cannot
    decide and the division sequence must (ties to even)."""
    rng = np.random.default_rng(64)
    M, K = 256, 384
    j = rng.integers(16, 32, size=(M, K))
    e = rng.integers(-6, 5, size=(M, K))
    sign = rng.choice([-1.0, 1.0], size=(M, K))
    f = (sign * 6.0 * j / 16.0 * np.exp2(e)).astype(np.float32)
    bits = synth.f32_to_bf16_bits(f)
    # Most row blocks' amaxes are such ties.
    b = np.abs(f).reshape(M, K // 16, 16).max(axis=2) / 6.0
    sig = b / np.exp2(np.floor(np.log2(b)))
    assert np.mean((sig * 16) % 2 == 1) > 0.3
    _nvfp4_case(bits, 2688.0, BOTH | (mxq.NVFP4_2D if two_d else 0), "ties")


@pytest.mark.parametrize("two_d", [False, True], ids=["1d", "2d"])
@pytest.mark.parametrize("log2_scale", [-97, -90], ids=["amax_2^-95", "amax_2^-88"])
def test_nvfp4_tiny_tensor_amax(two_d, log2_scale):
    """Tensor amaxes near 2^-95 (G below 2^-100: every block takes the
    division sequence) and 2^-88 (just above), with zero, subnormal and
    outlier blocks."""
    bits = _scaled_bits(synth.dbias(M=256, K=384, seed=65), 2.0 ** log2_scale)
    _nvfp4_case(bits, None, BOTH | (mxq.NVFP4_2D if two_d else 0), f"scale 2^{log2_scale}")


@pytest.mark.parametrize("two_d", [False, True], ids=["1d", "2d"])
def test_nvfp4_caller_amax_far_below_data(two_d):
    """Data near 2^100 with a caller amax of 2^-60: (b / 6) / G overflows to
    infinity and every block saturates to code 0x7E."""
    bits = _scaled_bits(synth.nvfp4(M=128, K=256, seed=66), 2.0 ** 100)
    _nvfp4_case(bits, 2.0 ** -60, BOTH | (mxq.NVFP4_2D if two_d else 0), "amax 2^-60")


def test_sharded_helpers_single_rank_nccl():
    """The sharded helpers through NCCL on a one-rank group (this box has one
    GPU): the collectives pass device tensors and the results equal the
    unsharded calls."""
    import socket
    import torch.distributed as dist
    from fp4_quantization_gb300 import sharded
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        bits = synth.nvfp4(M=256, K=512, seed=78)
        x = to_device(bits)
        got = sharded.nvfp4_quantize_transpose_sharded(x, BOTH)
        want = mxq.nvfp4_quantize_transpose(x, BOTH)
        for key in ("q_row", "s_row", "q_t", "s_t", "global_scale"):
            assert torch.equal(got[key], want[key]), key
        got = sharded.mx_quantize_rowcol_dbias_sharded(x, BOTH)
        want = mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS)
        for key in want:
            assert torch.equal(got[key], want[key]), key
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("M,K", [(96, 256), (1, 8), (333, 72), (4100, 1000), (5, 40000)])
def test_bf16_amax(M, K):
    """Blocks of whole rows: one block, several with a partial last one
    (4100 rows of 2000 bytes), and rows longer than a block's share."""
    bits = synth.nvfp4(M=max(M, 16), K=max(K, 16), seed=48)[:M, :K].copy()
    got = host(mxq.bf16_amax(to_device(bits)))[0]
    assert got == np.float32(oracle.bf16_amax(bits))


@pytest.mark.parametrize("where", ["first", "last"])
def test_bf16_amax_strided_window(where):
    """ldx > K (a column window of a wider matrix), the largest magnitude in
    the first or the last row, and larger values outside the window that
    must not count."""
    full = synth.nvfp4(M=4100, K=1064, seed=49)
    full[:, 1000:] = 0x7F00                     # 1.7e38 outside the window
    r = 0 if where == "first" else 4099
    full[r, 37] = 0xC700                        # -32768 inside it
    window = torch.from_numpy(full.view(np.int16)).view(torch.bfloat16).cuda()[:, 8:1000]
    got = host(mxq.bf16_amax(window))[0]
    assert got == np.float32(oracle.bf16_amax(full[:, 8:1000].copy())) == np.float32(32768.0)


def test_empty_inputs():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    out = mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS)
    torch.cuda.synchronize()
    assert out["q_row"].numel() == 0 and torch.all(out["dbias"] == 0)
    out = mxq.nvfp4_quantize_transpose(x, BOTH)
    assert host(out["global_scale"])[0] == 0.0
    amax = torch.tensor([5376.0], device="cuda")
    out = mxq.nvfp4_quantize_transpose(x, BOTH, amax=amax)
    assert host(out["global_scale"])[0] == 2.0
    assert host(mxq.bf16_amax(x))[0] == 0.0


def test_device_side_errors():
    bits = synth.rowcol(M=64, K=128, seed=49)
    x = to_device(bits)
    big = torch.empty(64 * 129, dtype=torch.bfloat16, device="cuda")
    shifted = big[1:1 + 64 * 128].view(64, 128)            # 2-byte offset: misaligned
    with pytest.raises(mxq.MxqError) as e:
        mxq.mx_quantize_rowcol(shifted, BOTH)
    assert e.value.status == 3
    with pytest.raises(mxq.MxqError) as e:
        mxq.mx_quantize_rowcol(x, BOTH | mxq.DBIAS, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 5
    with pytest.raises(mxq.MxqError) as e:
        mxq.nvfp4_quantize_transpose(x, BOTH, workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 5


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing completes gives up after its limit and reports
    MXQ_DEVERR_TIMEOUT; the next quantization still runs correctly."""
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mxq.mxq_selftest_bounded_wait(20_000_000, dev_err)    # 20 ms
    torch.cuda.synchronize()
    assert dev_err.item() == mxq.DEVERR_TIMEOUT
    bits = synth.plain_small()
    out = mxq.mx_quantize_rowcol(to_device(bits), BOTH)
    ref = oracle.mx_quantize(bits, BOTH)
    assert_equal_bytes(host(out["q_col"]), ref["q_col"], "after timeout")


def test_non_default_stream():
    bits = synth.rowcol(M=256, K=256, seed=50)
    x = to_device(bits)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = mxq.mx_quantize_rowcol(x, BOTH)
    s.synchronize()
    ref = oracle.mx_quantize(bits, BOTH)
    assert_equal_bytes(host(out["q_row"]), ref["q_row"], "stream q_row")


def test_two_launch_paths_back_to_back():
    """The dbias finalize and the NVFP4 quantize after its amax pass are
    launched as programmatic dependents of the grid before them: calls on two
    inputs, alternated without synchronising and sharing one workspace, each
    see only their own first grid's results."""
    a_bits = synth.dbias(M=2048, K=1024, seed=60)
    b_bits = synth.dbias(M=2048, K=1024, seed=61)
    a, b = to_device(a_bits), to_device(b_bits)
    flags = BOTH | mxq.DBIAS
    ws = torch.empty(mxq.mxq_workspace_bytes(mxq.OP_ROWCOL, 2048, 1024, flags), dtype=torch.uint8,
                     device="cuda")
    out_a = mxq.mx_quantize_rowcol(a, flags, workspace=ws)
    out_b = mxq.mx_quantize_rowcol(b, flags, workspace=ws)
    for _ in range(3):
        mxq.mx_quantize_rowcol(a, flags, workspace=ws, **out_a)
        mxq.mx_quantize_rowcol(b, flags, workspace=ws, **out_b)
    torch.cuda.synchronize()
    for bits, out in ((a_bits, out_a), (b_bits, out_b)):
        ref = oracle.mx_quantize(bits, flags)
        for key in ("q_row", "s_row", "q_col", "s_col"):
            assert_equal_bytes(host(out[key]), ref[key], f"back-to-back dbias {key}")
        err = np.abs(host(out["dbias"]).astype(np.float64) - ref["dbias"].astype(np.float64))
        assert np.all(err <= _dbias_tolerance(bits)), f"back-to-back dbias max err {err.max()}"

    c_bits = synth.nvfp4(M=512, K=1024, seed=62)
    d_f32 = synth.bf16_bits_to_f32(synth.nvfp4(M=512, K=1024, seed=63)) * np.float32(8.0)
    d_bits = (d_f32.view(np.uint32) >> 16).astype(np.uint16)   # exact: x 8 keeps bf16 values
    c, d = to_device(c_bits), to_device(d_bits)
    nws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out_c = mxq.nvfp4_quantize_transpose(c, BOTH, workspace=nws)
    out_d = mxq.nvfp4_quantize_transpose(d, BOTH, workspace=nws)
    for _ in range(3):
        mxq.nvfp4_quantize_transpose(c, BOTH, workspace=nws, **out_c)
        mxq.nvfp4_quantize_transpose(d, BOTH, workspace=nws, **out_d)
    torch.cuda.synchronize()
    for bits, out in ((c_bits, out_c), (d_bits, out_d)):
        ref = oracle.nvfp4_quantize(bits)
        assert host(out["global_scale"])[0] == np.float32(ref["global_scale"])
        for key in ("q_row", "s_row", "q_t", "s_t"):
            assert_equal_bytes(host(out[key]), ref[key], f"back-to-back nvfp4 {key}")
