"""Pins for the oracle's whole-matrix quantizers (CPU only).

Each test checks the oracle against something fixed from outside its code:
hand-worked blocks, exact round trips, the half-step error bound of
round-to-nearest, transpose symmetry between the rowwise and colwise
layouts, closed forms on bf16 bit patterns, exact sums (math.fsum), and
alternative closed forms of the activations.
"""
import math

import numpy as np
import pytest

import oracle
import synth

from test_oracle_formats import E2M1, E4M3


def bf16(values):
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(values, dtype=np.float32)
    bits = synth.f32_to_bf16_bits(f)
    back = synth.bf16_bits_to_f32(bits)
    assert np.array_equal(back, f, equal_nan=True), "value not exactly representable in bf16"
    return bits


def f32(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# --------------------------------------------------------------------------
# MXFP8
# --------------------------------------------------------------------------

def test_mx_hand_worked_blocks():
    """Three 1x32 blocks worked by hand (rows 0-2 of a 32x32 matrix)."""
    x = np.zeros((32, 32), np.float32)
    # Row 0: amax 3.0 -> floor(log2 3) = 1 -> e = -7 -> code 120, v = 128 x.
    x[0, :5] = [3.0, 0.10009765625, 17 / 128, 19 / 128, -0.30078125]
    # Row 1: amax 1.9921875 -> floor(log2) = 0 -> e = -8 -> code 119, v = 256 x.
    x[1, :6] = [1.9921875, 1.75, 2.0 ** -16, 3 * 2.0 ** -18, 2.0 ** -18, -(2.0 ** -18)]
    # Row 2: amax 2^-128 (bf16 subnormal) -> e clamps to -127 -> code 0, v = 2^127 x.
    x[2, :3] = [2.0 ** -128, -3 * 2.0 ** -131, 2.0 ** -133]
    out = oracle.mx_quantize(bf16(x), oracle.ROWWISE)
    assert list(out["s_row"][:3, 0]) == [120, 119, 0]
    assert list(out["q_row"][0, :5]) == [0x7C, 0x55, 0x58, 0x5A, 0xE2]
    assert list(out["q_row"][1, :6]) == [0x7E, 0x7E, 0x02, 0x02, 0x00, 0x80]
    assert list(out["q_row"][2, :3]) == [0x30, 0xA4, 0x08]
    # The untouched zeros of those rows stay zero; rows 3.. are all-zero blocks.
    assert not out["q_row"][0, 5:].any() and not out["q_row"][3:].any()
    assert not out["s_row"][3:].any()
    # Largest finite bf16 as amax -> code 246.
    big = np.zeros((32, 32), np.uint16)
    big[0, 0] = 0x7F7F
    assert oracle.mx_quantize(big, oracle.ROWWISE)["s_row"][0, 0] == 246


def test_mx_transpose_symmetry():
    """Colwise outputs of x are the rowwise outputs of x transposed."""
    x = synth.dbias(M=96, K=160, seed=21)
    a = oracle.mx_quantize(x, oracle.ROWWISE | oracle.COLWISE)
    b = oracle.mx_quantize(np.ascontiguousarray(x.T), oracle.ROWWISE | oracle.COLWISE)
    np.testing.assert_array_equal(a["q_col"], b["q_row"])
    np.testing.assert_array_equal(a["s_col"], b["s_row"])
    np.testing.assert_array_equal(a["q_row"], b["q_col"])
    np.testing.assert_array_equal(a["s_row"], b["s_col"])


def test_mx_scale_closed_form():
    """Scale code = max(0, exponent field of the block's largest |x| - 8),
    computed here from bf16 bit patterns without any float arithmetic."""
    x = synth.dbias(M=128, K=256, seed=22)
    out = oracle.mx_quantize(x, oracle.ROWWISE | oracle.COLWISE)
    mag = (x & 0x7FFF).astype(np.int64)
    row_max = mag.reshape(128, 8, 32).max(axis=2)
    col_max = mag.reshape(4, 32, 256).max(axis=1).T
    np.testing.assert_array_equal(out["s_row"], np.maximum(0, (row_max >> 7) - 8))
    np.testing.assert_array_equal(out["s_col"], np.maximum(0, (col_max >> 7) - 8))


def _dequant_error_ok(xv, q, scale_code):
    """Round-to-nearest bound: |x - value(q) 2^e| <= half a step of q's
    binade times 2^e, for every element whose scaled magnitude is at most
    464 (448 plus half a step); saturated elements above that are skipped."""
    e = scale_code.astype(np.int64) - 127
    v = np.ldexp(xv, -e)
    deq = E4M3[q]
    code_exp = (q.astype(np.int64) >> 3) & 0xF
    step = np.where(code_exp == 0, 2.0 ** -9, np.exp2(code_exp - 10.0))
    in_range = np.abs(v) <= 464.0
    err = np.abs(v - deq)
    return np.all(err[in_range] <= 0.5 * step[in_range]), np.all(np.abs(deq[~in_range]) == 448.0)


def test_mx_half_step_bound_and_monotone():
    x = synth.dbias(M=256, K=256, seed=23)
    out = oracle.mx_quantize(x, oracle.ROWWISE | oracle.COLWISE)
    xv = f32(x)
    s_rep = np.repeat(out["s_row"], 32, axis=1)
    bound_ok, sat_ok = _dequant_error_ok(xv, out["q_row"], s_rep)
    assert bound_ok and sat_ok
    s_rep_c = np.repeat(out["s_col"], 32, axis=1)
    bound_ok, sat_ok = _dequant_error_ok(xv.T, out["q_col"], s_rep_c)
    assert bound_ok and sat_ok
    # Within a block, the dequantized values keep the order of the inputs.
    blocks_x = xv.reshape(256, 8, 32)
    blocks_q = E4M3[out["q_row"]].reshape(256, 8, 32)
    order = np.argsort(blocks_x, axis=2, kind="stable")
    deq_sorted = np.take_along_axis(blocks_q, order, axis=2)
    assert np.all(np.diff(deq_sorted, axis=2) >= 0)


def test_mx_exact_round_trip():
    """Blocks whose values are E4M3 values times 2^s, with one element at
    448 * 2^s, dequantize exactly (the scale comes out as 2^s)."""
    rng = np.random.default_rng(3)
    finite_pos = [c for c in range(0x7F) if E4M3[c] * 1 == E4M3[c]]
    rows = []
    shifts = [-120, -40, -9, -1, 0, 3, 17, 100, 118]
    for s in shifts:
        codes = rng.choice(finite_pos, size=32)
        codes[0] = 0x7E
        signs = rng.choice([-1.0, 1.0], size=32)
        rows.append(signs * np.ldexp(E4M3[codes], s))
    x = np.array(rows)
    out = oracle.mx_quantize(bf16(np.pad(x, ((0, 32 - len(shifts)), (0, 0)))), oracle.ROWWISE)
    for i, s in enumerate(shifts):
        assert out["s_row"][i, 0] == s + 127
        np.testing.assert_array_equal(np.ldexp(E4M3[out["q_row"][i]], s), x[i])


def test_mx_special_blocks_small_workload():
    """The all-zero tile and the 2^-130-scaled tile of the 128x256 workload."""
    x = synth.plain_small()
    out = oracle.mx_quantize(x, oracle.ROWWISE | oracle.COLWISE)
    assert not out["s_row"][0:32, 0].any() and not out["q_row"][0:32, 0:32].any()
    assert not out["s_col"][0:32, 0].any() and not out["q_col"][0:32, 0:32].any()
    # Subnormal tile: every scale clamps to code 0, so codes are E4M3(x * 2^127).
    assert not out["s_row"][32:64, 2].any() and not out["s_col"][64:96, 1].any()
    v = np.ldexp(f32(x[32:64, 64:96]), 127)
    np.testing.assert_array_equal(out["q_row"][32:64, 64:96], oracle.e4m3_encode(v).reshape(32, 32))
    np.testing.assert_array_equal(out["q_col"][64:96, 32:64], oracle.e4m3_encode(v.T).reshape(32, 32))


def test_mx_empty_and_bad_shapes():
    out = oracle.mx_quantize(np.zeros((0, 64), np.uint16), oracle.ROWWISE | oracle.DBIAS)
    assert out["q_row"].shape == (0, 64)
    assert np.all(out["dbias"] == 0)
    with pytest.raises(ValueError):
        oracle.mx_quantize(np.zeros((32, 48), np.uint16))
    with pytest.raises(ValueError):
        oracle.mx_quantize(np.zeros((40, 64), np.uint16))


def test_mx_window_view_matches_full():
    """A strided window of a larger matrix gives the same blocks as the full
    matrix (the sampled full-size GPU checks rely on this)."""
    x = synth.rowcol(M=128, K=320, seed=7)
    full = oracle.mx_quantize(x)
    w = oracle.mx_quantize(x[32:96, 64:256])
    np.testing.assert_array_equal(w["q_row"], full["q_row"][32:96, 64:256])
    np.testing.assert_array_equal(w["s_row"], full["s_row"][32:96, 2:8])
    np.testing.assert_array_equal(w["q_col"], full["q_col"][64:256, 32:96])
    np.testing.assert_array_equal(w["s_col"], full["s_col"][64:256, 1:3])


# --------------------------------------------------------------------------
# dbias
# --------------------------------------------------------------------------

def test_dbias_is_exact_column_sum():
    x = synth.dbias(M=320, K=96, seed=24)
    out = oracle.mx_quantize(x, oracle.DBIAS)
    xv = f32(x)
    want = np.array([np.float32(math.fsum(xv[:, k])) for k in range(96)], np.float32)
    np.testing.assert_array_equal(out["dbias"], want)


# --------------------------------------------------------------------------
# Activations
# --------------------------------------------------------------------------

def _ulp32(v):
    return np.spacing(np.abs(np.float32(v))).astype(np.float64)


def test_gelu_identities():
    rng = np.random.default_rng(8)
    xs = np.concatenate([rng.standard_normal(2000) * 3, [0.0, 1e-30, 5.0, -5.0, 20.0, -20.0]]).astype(np.float32)
    assert oracle.gelu_tanh(0.0) == 0.0
    for x in xs:
        g, gm = oracle.gelu_tanh(x), oracle.gelu_tanh(-x)
        # 0.5 x (1 + tanh(u)) with u odd in x: gelu(x) - gelu(-x) = x.
        assert abs((g - gm) - float(x)) <= _ulp32(g) + _ulp32(gm) + 1e-45
        # Same function through the logistic form x / (1 + exp(-2u)).
        xd = float(x)
        u = math.sqrt(2 / math.pi) * (xd + 0.044715 * xd ** 3)
        alt = xd / (1.0 + math.exp(-2 * u)) if u > -350 else 0.0
        assert abs(g - alt) <= _ulp32(alt) + 1e-45


def test_swiglu_identities():
    rng = np.random.default_rng(9)
    gs = (rng.standard_normal(2000) * 2).astype(np.float32)
    us = rng.standard_normal(2000).astype(np.float32)
    for g, u in zip(gs, us):
        s, sm = oracle.swiglu(g, 1.0), oracle.swiglu(-g, 1.0)
        assert abs((s - sm) - float(g)) <= _ulp32(s) + _ulp32(sm)     # silu(g) - silu(-g) = g
        # Linear in the up operand; doubling is exact.
        assert oracle.swiglu(g, 2 * u) == 2 * oracle.swiglu(g, u)
        # silu through the tanh form g (1 + tanh(g/2)) / 2.
        alt = float(g) * (1 + math.tanh(float(g) / 2)) / 2 * float(u)
        assert abs(oracle.swiglu(g, u) - alt) <= _ulp32(alt) + 1e-45


def test_activation_quantize_composes():
    """GELU and SwiGLU quantization = activation per element, then the plain
    block rule built here from the (separately pinned) scalar encoders."""
    x = synth.gelu(M=64, K=64, seed=10)
    out = oracle.mx_quantize(x, oracle.ROWWISE | oracle.COLWISE, act=oracle.ACT_GELU_TANH)
    y = np.array([[oracle.gelu_tanh(v) for v in row] for row in synth.bf16_bits_to_f32(x)])
    _check_blocks(y, out)
    xg = synth.swiglu(M=64, N=64, seed=11)
    outg = oracle.mx_quantize_swiglu(xg, 64)
    xf = synth.bf16_bits_to_f32(xg)
    yg = np.array([[oracle.swiglu(xf[m, n], xf[m, 64 + n]) for n in range(64)] for m in range(64)])
    _check_blocks(yg, outg)


def _richardson(f, x, h):
    """Derivative of f at x by central differences with one Richardson step
    (error O(h^4)), in float64."""
    d1 = (f(x + h) - f(x - h)) / (2 * h)
    d2 = (f(x + h / 2) - f(x - h / 2)) / h
    return (4 * d2 - d1) / 3


def _gelu64(x):
    return 0.5 * x * (1 + np.tanh(np.sqrt(2 / np.pi) * (x + 0.044715 * x ** 3)))


def _silu64(x):
    return x / (1 + np.exp(-x))


def test_activation_derivatives():
    """dgelu / dsilu against numerical differentiation of the functions
    themselves, plus the values the closed forms fix: 1/2 at 0, 1 far right,
    0 far left (the GELU derivative dips just below 0 before it)."""
    rng = np.random.default_rng(16)
    xs = np.concatenate([rng.standard_normal(3000) * 3,
                         np.linspace(-6, 6, 241)]).astype(np.float32)
    for f64, d_or in ((_gelu64, oracle.dgelu_tanh), (_silu64, oracle.dsilu)):
        for x in xs:
            xd = float(x)
            want = _richardson(f64, xd, 1e-2 * max(1.0, abs(xd)))
            got = d_or(x)
            assert abs(got - want) <= 2e-7 * max(1.0, abs(want)), (d_or.__name__, xd, got, want)
    assert oracle.dgelu_tanh(0.0) == 0.5 and oracle.dsilu(0.0) == 0.5
    assert oracle.dgelu_tanh(20.0) == 1.0 and oracle.dsilu(40.0) == 1.0
    assert abs(oracle.dgelu_tanh(-20.0)) < 1e-30 and abs(oracle.dsilu(-110.0)) < 1e-30
    assert min(oracle.dgelu_tanh(x) for x in np.linspace(-3, -1, 81)) < 0   # the dip


def test_geglu_reduces_to_gelu():
    """GeGLU with up = 1 is GELU of the gate (the pinned GELU path), bit for
    bit; up = 2 doubles every value, so the codes stay and each scale code
    moves up by one."""
    gate = synth.gelu(M=64, K=96, seed=17)
    ones = np.full_like(gate, 0x3F80)                      # bf16 1.0
    twos = np.full_like(gate, 0x4000)                      # bf16 2.0
    ref = oracle.mx_quantize(gate, oracle.ROWWISE | oracle.COLWISE, act=oracle.ACT_GELU_TANH)
    got = oracle.mx_quantize_gated(np.hstack([gate, ones]), 96, act=oracle.ACT_GELU_TANH)
    for key in ref:
        np.testing.assert_array_equal(got[key], ref[key])
    dbl = oracle.mx_quantize_gated(np.hstack([gate, twos]), 96, act=oracle.ACT_GELU_TANH)
    np.testing.assert_array_equal(dbl["q_row"], ref["q_row"])
    nz = ref["s_row"] > 0
    np.testing.assert_array_equal(dbl["s_row"][nz], ref["s_row"][nz] + 1)


def test_dact_quantize_composes():
    """y = grad * act'(x) with grad a power of two (so the product is the
    exactly scaled fp32 derivative), then the block rule built here from the
    pinned encoders; dbias = exact column sums of y."""
    x = synth.gelu(M=64, K=64, seed=18)
    rng = np.random.default_rng(19)
    gvals = rng.choice(np.array([1.0, -1.0, 2.0, -0.5, 0.25, 4.0], np.float32), size=(64, 64))
    grad = bf16(gvals)
    xf = synth.bf16_bits_to_f32(x)
    for act, d in ((oracle.ACT_GELU_TANH, oracle.dgelu_tanh), (oracle.ACT_SILU, oracle.dsilu)):
        out = oracle.mx_quantize_dact(grad, x, act, oracle.ROWWISE | oracle.COLWISE | oracle.DBIAS)
        y = np.array([[np.float32(gvals[m, k]) * np.float32(d(xf[m, k])) for k in range(64)]
                      for m in range(64)], np.float32)
        _check_blocks(y.astype(np.float64), out)
        want = np.array([np.float32(math.fsum(y[:, k].astype(np.float64))) for k in range(64)])
        np.testing.assert_array_equal(out["dbias"], want)


def test_dgated_halves():
    """With grad = 1 and up = 1, the d-gate half of the backward gated output
    is act'(gate) (the pinned dact path) and the d-up half is act(gate) (the
    pinned gated forward with up = 1); the halves are whole 32-column blocks
    rowwise and whole code rows colwise."""
    gate = synth.gelu(M=64, K=64, seed=20)
    ones = np.full_like(gate, 0x3F80)
    x = np.hstack([gate, ones])
    for act in (oracle.ACT_SILU, oracle.ACT_GELU_TANH):
        out = oracle.mx_quantize_dgated(ones, x, 64, act)
        dact = oracle.mx_quantize_dact(ones, gate, act)
        fwd = oracle.mx_quantize_gated(x, 64, act=act)
        np.testing.assert_array_equal(out["q_row"][:, :64], dact["q_row"])
        np.testing.assert_array_equal(out["s_row"][:, :2], dact["s_row"])
        np.testing.assert_array_equal(out["q_col"][:64], dact["q_col"])
        np.testing.assert_array_equal(out["s_col"][:64], dact["s_col"])
        np.testing.assert_array_equal(out["q_row"][:, 64:], fwd["q_row"])
        np.testing.assert_array_equal(out["s_row"][:, 2:], fwd["s_row"])
        np.testing.assert_array_equal(out["q_col"][64:], fwd["q_col"])
        np.testing.assert_array_equal(out["s_col"][64:], fwd["s_col"])


def test_dgated_products_compose():
    """The gated backward with grad and up that vary per element: powers of
    two (grad in {+-0.5, 2, 4}, up in {+-0.25, 2, 8}), so each product is an
    exact rescaling of the separately pinned scalar.  Rebuilt here:
    d gate = grad * up * act'(gate) and d up = grad * act(gate), then the
    blocks from the pinned encoders.  Dropping up or grad from either half,
    or taking act'(up), changes these blocks."""
    M, N = 64, 64
    gate = synth.gelu(M=M, K=N, seed=21)
    rng = np.random.default_rng(22)
    gvals = rng.choice(np.array([0.5, -0.5, 2.0, 4.0], np.float32), size=(M, N))
    uvals = rng.choice(np.array([0.25, -0.25, 2.0, 8.0], np.float32), size=(M, N))
    grad, up = bf16(gvals), bf16(uvals)
    x = np.hstack([gate, up])
    gf = synth.bf16_bits_to_f32(gate)
    for act, dfn, fn in ((oracle.ACT_SILU, oracle.dsilu, lambda v: oracle.swiglu(v, 1.0)),
                         (oracle.ACT_GELU_TANH, oracle.dgelu_tanh, oracle.gelu_tanh)):
        out = oracle.mx_quantize_dgated(grad, x, N, act)
        y = np.empty((M, 2 * N), np.float32)
        for m in range(M):
            for n in range(N):
                y[m, n] = gvals[m, n] * uvals[m, n] * np.float32(dfn(gf[m, n]))
                y[m, N + n] = gvals[m, n] * np.float32(fn(gf[m, n]))
        _check_blocks(y.astype(np.float64), out)


def _check_blocks(y, out):
    M, K = y.shape
    for m in range(M):
        for kb in range(K // 32):
            blk = y[m, kb * 32:(kb + 1) * 32]
            code = oracle.e8m0_code([np.abs(blk).max()])[0]
            assert out["s_row"][m, kb] == code
            np.testing.assert_array_equal(out["q_row"][m, kb * 32:(kb + 1) * 32],
                                          oracle.e4m3_encode(np.ldexp(blk, 127 - int(code))))
    for k in range(K):
        for mb in range(M // 32):
            blk = y[mb * 32:(mb + 1) * 32, k]
            code = oracle.e8m0_code([np.abs(blk).max()])[0]
            assert out["s_col"][k, mb] == code
            np.testing.assert_array_equal(out["q_col"][k, mb * 32:(mb + 1) * 32],
                                          oracle.e4m3_encode(np.ldexp(blk, 127 - int(code))))


# --------------------------------------------------------------------------
# NVFP4
# --------------------------------------------------------------------------

def test_nvfp4_hand_worked():
    """Tensor amax 2688 makes the global scale exactly 1."""
    x = np.zeros((16, 16), np.float32)
    x[0, 0] = 2688.0            # block amax 2688: s = E4M3(448) = 0x7E, d = 448, 2688/448 = 6
    x[1, :12] = [6, 3, -1.5, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.0, 1]   # amax 6: s = 1.0 (0x38)
    x[2, :2] = [3.0, 1.5]       # amax 3: s = E4M3(0.5) = 0x30, d = 0.5, inv = 2
    x[2, 2] = 0.30078125        # * 2 = 0.6015625 -> nearest E2M1 0.5 (code 1)
    out = oracle.nvfp4_quantize(bf16(x), flags=oracle.ROWWISE)
    assert out["global_scale"] == 1.0
    assert list(out["s_row"][:3, 0]) == [0x7E, 0x38, 0x30]
    assert out["q_row"][0, 0] == 0x07                        # 6 -> code 7, low nibble
    row1 = [0x7, 0x5, 0xB, 0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x8, 0x2, 0, 0, 0, 0]
    assert list(out["q_row"][1]) == [row1[2 * i] | (row1[2 * i + 1] << 4) for i in range(8)]
    assert out["q_row"][2, 0] == (0x7 | (0x5 << 4))         # 3*2 = 6 -> 7, 1.5*2 = 3 -> 5
    assert out["q_row"][2, 1] == 0x1                         # 0.6015625 -> 0.5
    assert not out["s_row"][3:].any() and not out["q_row"][3:].any()


def test_nvfp4_zero_tensor():
    x = np.zeros((32, 32), np.uint16)
    x[5, 7] = 0x8000              # -0
    out = oracle.nvfp4_quantize(x)
    assert out["global_scale"] == 0.0
    assert not out["s_row"].any() and not out["s_t"].any()
    assert out["q_row"][5, 3] == 0x80 and out["q_t"][7, 2] == 0x80   # sign of -0 kept
    assert np.count_nonzero(out["q_row"]) == 1 and np.count_nonzero(out["q_t"]) == 1


def test_nvfp4_transpose_symmetry_and_bound():
    x = synth.nvfp4(M=96, K=128, seed=12)
    a = oracle.nvfp4_quantize(x)
    b = oracle.nvfp4_quantize(np.ascontiguousarray(x.T), tensor_amax=oracle.bf16_amax(x))
    np.testing.assert_array_equal(a["q_t"], b["q_row"])
    np.testing.assert_array_equal(a["s_t"], b["s_row"])
    # Error bound: |x - value(q) d| <= half an E2M1 step of q's binade times
    # d (plus the fp32 rounding of x * inv), except where x * inv exceeds 6.
    xv = f32(x)
    G = a["global_scale"]
    assert G == np.float32(np.float32(oracle.bf16_amax(x)) / np.float32(2688.0))
    lo = a["q_row"] & 0xF
    hi = a["q_row"] >> 4
    codes = np.stack([lo, hi], axis=2).reshape(96, 128)
    d = np.repeat(E4M3[a["s_row"]].astype(np.float32) * np.float32(G), 16, axis=1).astype(np.float64)
    deq = E2M1[codes] * d
    e = (codes >> 1) & 3
    step = np.where(e == 0, 0.5, np.exp2(e - 2.0)) * d
    in_range = np.abs(xv) <= 6.5 * d
    err = np.abs(xv - deq) - 0.5 * step - np.abs(xv) * 2.0 ** -22
    assert np.all(err[in_range] <= 0)


# --------------------------------------------------------------------------
# NVFP4 2D (16x16 blocks)
# --------------------------------------------------------------------------

TWO_D = oracle.NVFP4_2D


def _unpack(q):
    """Packed E2M1 bytes [R, C/2] -> codes [R, C] (element 2i in the low nibble)."""
    return np.stack([q & 0xF, q >> 4], axis=2).reshape(q.shape[0], -1)


def test_nvfp4_2d_hand_worked():
    """Tensor amax 2688 makes G = 1.  Block (0, 0) has its amax 6 in row 0, so
    every row of the block is scaled by s = 1.0 (0x38, inv 1): 0.5 in row 5
    stays 0.5 (code 1), where a 1x16 block of that row alone (amax 0.5,
    d = E4M3(0.5 / 6) = 0.0859375, 0.5 / d = 5.82 -> 6) gives it code 7.  Block (0, 1) is all zero;
    block (1, 0) holds the tensor amax: s = 0x7E (448), inv = 1/448."""
    x = np.zeros((32, 32), np.float32)
    x[0, 0] = 6.0
    x[5, 3] = 0.5
    x[9, 15] = -1.5
    x[15, 8] = 3.0
    x[16, 0] = 2688.0
    x[20, 4] = 896.0            # / 448 = 2 -> code 4
    x[31, 15] = -0.0
    out = oracle.nvfp4_quantize(bf16(x), tensor_amax=2688.0, flags=3 | TWO_D)
    assert out["global_scale"] == 1.0
    s_row, s_t = out["s_row"], out["s_t"]
    assert np.all(s_row[:16, 0] == 0x38) and np.all(s_row[:16, 1] == 0)
    assert np.all(s_row[16:, 0] == 0x7E) and np.all(s_row[16:, 1] == 0)
    assert np.all(s_t[:16, 0] == 0x38) and np.all(s_t[:16, 1] == 0x7E)
    assert np.all(s_t[16:, :] == 0)
    c = _unpack(out["q_row"])
    assert c[0, 0] == 0x7 and c[5, 3] == 0x1 and c[9, 15] == 0xB and c[15, 8] == 0x5
    assert c[16, 0] == 0x7 and c[20, 4] == 0x4 and c[31, 15] == 0x8
    assert np.count_nonzero(c) == 7
    one_d = oracle.nvfp4_quantize(bf16(x), tensor_amax=2688.0, flags=oracle.ROWWISE)
    assert _unpack(one_d["q_row"])[5, 3] == 0x7        # the 1x16 reading differs


def test_nvfp4_2d_transposed_output_is_the_transpose():
    """Each element takes its block's scale in both outputs, so the
    transposed codes are the rowwise codes transposed, and the transposed
    scale of (k, block mb) is the rowwise scale of (rows of mb, k / 16)."""
    x = synth.nvfp4(M=96, K=160, seed=13)
    out = oracle.nvfp4_quantize(x, flags=3 | TWO_D)
    np.testing.assert_array_equal(_unpack(out["q_t"]), _unpack(out["q_row"]).T)
    per_block = out["s_row"][::16, :]                       # [M/16, K/16]
    np.testing.assert_array_equal(out["s_row"], np.repeat(per_block, 16, axis=0))
    np.testing.assert_array_equal(out["s_t"], np.repeat(per_block.T, 16, axis=0))


def test_nvfp4_2d_transpose_symmetry():
    """The 2D blocks of x^T are the transposed blocks of x."""
    x = synth.nvfp4(M=64, K=96, seed=14)
    a = oracle.nvfp4_quantize(x, flags=3 | TWO_D)
    b = oracle.nvfp4_quantize(np.ascontiguousarray(x.T), tensor_amax=oracle.bf16_amax(x),
                              flags=3 | TWO_D)
    np.testing.assert_array_equal(a["q_t"], b["q_row"])
    np.testing.assert_array_equal(a["s_t"], b["s_row"])
    np.testing.assert_array_equal(a["q_row"], b["q_t"])


def test_nvfp4_2d_reduces_to_1d_on_repeated_rows_and_columns():
    """When the 16 rows of every block are equal, a 16x16 block has the amax
    of each of its 1x16 rows, so the 2D rowwise output equals the 1D one;
    likewise for the transposed output when the 16 columns are equal."""
    base = synth.nvfp4(M=64, K=128, seed=15)
    rows = np.repeat(base[::16], 16, axis=0)               # rows repeat in 16-row groups
    A = oracle.bf16_amax(rows)
    two = oracle.nvfp4_quantize(rows, tensor_amax=A, flags=3 | TWO_D)
    one = oracle.nvfp4_quantize(rows, tensor_amax=A, flags=3)
    np.testing.assert_array_equal(two["q_row"], one["q_row"])
    np.testing.assert_array_equal(two["s_row"], one["s_row"])
    cols = np.repeat(base[:, ::16], 16, axis=1)            # columns repeat in 16-column groups
    A = oracle.bf16_amax(cols)
    two = oracle.nvfp4_quantize(cols, tensor_amax=A, flags=3 | TWO_D)
    one = oracle.nvfp4_quantize(cols, tensor_amax=A, flags=3)
    np.testing.assert_array_equal(two["q_t"], one["q_t"])
    np.testing.assert_array_equal(two["s_t"], one["s_t"])


def test_mx_rceil_blocks_never_saturate():
    """With the ceil rule every block's largest element maps to at most 448
    (no saturation), the scale is the pinned ceil code of the block amax, and
    the codes are the pinned E4M3 encoder's."""
    x = synth.dbias(M=64, K=96, seed=23)
    out = oracle.mx_quantize(x, oracle.ROWWISE | oracle.COLWISE | oracle.SCALE_RCEIL)
    y = f32(x)
    for m in range(64):
        for kb in range(3):
            blk = y[m, kb * 32:(kb + 1) * 32]
            code = oracle.e8m0_code_rceil([np.abs(blk).max()])[0]
            assert out["s_row"][m, kb] == code
            v = np.ldexp(blk, 127 - int(code))
            assert np.abs(v).max() <= 448.0
            np.testing.assert_array_equal(out["q_row"][m, kb * 32:(kb + 1) * 32], oracle.e4m3_encode(v))
    for k in range(96):
        for mb in range(2):
            blk = y[mb * 32:(mb + 1) * 32, k]
            code = oracle.e8m0_code_rceil([np.abs(blk).max()])[0]
            assert out["s_col"][k, mb] == code
            np.testing.assert_array_equal(out["q_col"][k, mb * 32:(mb + 1) * 32],
                                          oracle.e4m3_encode(np.ldexp(blk, 127 - int(code))))


def test_swizzle_matches_tile_reshape():
    """The tiled scale layout by its index formula equals the same layout
    built as a reshape: pad to [R', C'], view as [R'/128][4][32][C'/4][4]
    (tile row, row // 32 in tile, row % 32, tile column, column in tile) and
    order the axes (tile row, tile column, row % 32, row // 32, column); also
    a bijection of the padded positions."""
    rng = np.random.default_rng(24)
    for R, C in ((128, 4), (256, 12), (96, 6), (300, 17), (32, 1)):
        s = rng.integers(1, 255, size=(R, C), dtype=np.uint8)
        got = oracle.swizzle_scales(s)
        Rp, Cp = oracle.swizzled_shape(R, C)
        pad = np.zeros((Rp, Cp), np.uint8)
        pad[:R, :C] = s
        want = pad.reshape(Rp // 128, 4, 32, Cp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(Rp, Cp)
        np.testing.assert_array_equal(got, want)
        idx = np.arange(Rp * Cp).reshape(Rp, Cp) % 251 + 1
        assert np.array_equal(np.sort(oracle.swizzle_scales(idx.astype(np.uint8)).ravel()),
                              np.sort(idx.astype(np.uint8).ravel()))


def test_swizzled_quantize_is_the_row_major_result_retiled():
    x = synth.dbias(M=160, K=288, seed=25)
    plain = oracle.mx_quantize(x, 3)
    swz = oracle.mx_quantize(x, 3 | oracle.SCALE_SWIZZLED)
    np.testing.assert_array_equal(swz["q_row"], plain["q_row"])
    np.testing.assert_array_equal(swz["q_col"], plain["q_col"])
    np.testing.assert_array_equal(swz["s_row"], oracle.swizzle_scales(plain["s_row"]))
    np.testing.assert_array_equal(swz["s_col"], oracle.swizzle_scales(plain["s_col"]))
    assert swz["s_row"].shape == (256, 12) and swz["s_col"].shape == (384, 8)
