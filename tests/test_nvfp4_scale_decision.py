"""The rule the NVFP4 kernel uses to decide a block's E4M3 scale code without
a per-amax table, checked exhaustively over block amaxes against the recipe.

The recipe (TE PR #3291, "NVFP4 quantize-transpose" family; the fixed fp32
order in the kernel's header) is s = E4M3(RN(RN(b / 6) / G)).  The kernel
instead takes q = RN(b * K), K = RN(1 / RN(6 G)), and accepts the code of
the fp32 values 16 units in the last place below and above q when the two
agree; otherwise (and for every block when G < 2^-100) it runs the recipe's
divisions.  Restated here in numpy fp32 (IEEE round-to-nearest, like the
kernel's __fmul_rn / __frcp_rn), with the oracle's E4M3 encoder, over every
positive finite bf16 b: an accepted code must always be the recipe's.
"""
import numpy as np

import oracle

F32 = np.float32
ALL_B = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)   # every finite bf16 >= 0


def _decide(b, A):
    """(accepted, code_if_accepted, recipe_code) for block amaxes b, tensor amax A."""
    G = F32(A) / F32(2688.0)
    K = F32(1.0) / (F32(6.0) * G)
    with np.errstate(over="ignore"):
        q = (b * K).astype(np.float32)
        recipe = ((b / F32(6.0)).astype(np.float32) / G).astype(np.float32)
    bits = q.view(np.int32).astype(np.int64)
    lo = np.maximum(bits - 16, 0).astype(np.uint32).view(np.float32)
    hi = np.minimum(bits + 16, 0x7F7FFFFF).astype(np.uint32).view(np.float32)
    c_lo = oracle.e4m3_encode(lo.astype(np.float64))
    c_hi = oracle.e4m3_encode(hi.astype(np.float64))
    c_recipe = oracle.e4m3_encode(recipe.astype(np.float64))
    return c_lo == c_hi, c_lo, c_recipe


def _tensor_amaxes():
    """bf16 tensor amaxes from 2^-88 (G just above 2^-100) to the bf16 maximum:
    per binade a random significand and 1.3125 (A = 2688 * 2^k, G a power of
    two: the most exact ties)."""
    rng = np.random.default_rng(7)
    out = []
    for e in range(-88, 128, 3):
        for mant in (int(rng.integers(0, 128)), 0x28):
            out.append(np.array([((e + 127) << 7) | mant], np.uint32) << 16)
    out.append(np.array([0x7F7F << 16], np.uint32))
    return [float(a.view(np.float32)[0]) for a in out]


def test_fast_code_decision_never_wrong():
    wrong = 0
    deferred = {False: 0, True: 0}     # keyed by "G is a power of two"
    in_range = {False: 0, True: 0}
    for A in _tensor_amaxes():
        G = F32(A) / F32(2688.0)
        assert G >= F32(2.0 ** -100)
        pow2 = (G.view(np.uint32) & 0x7FFFFF) == 0
        ok, code, recipe = _decide(ALL_B, A)
        wrong += int(np.count_nonzero(ok & (code != recipe)))
        mask = ALL_B <= F32(A)
        in_range[bool(pow2)] += int(np.count_nonzero(mask))
        deferred[bool(pow2)] += int(np.count_nonzero(mask & ~ok))
    assert wrong == 0
    # Deferred blocks are rare for a generic G; with G a power of two the
    # recipe's quotient often lands exactly on a rounding boundary.
    assert deferred[False] / in_range[False] < 1e-3
    assert deferred[True] > 0


def test_exact_ties_are_deferred():
    """G = 1: b = 6 * 17/16 gives (b / 6) / G = 1.0625, halfway between the
    E4M3 values 1 and 1.125, and b = 28.5 gives 4.75, halfway between 4.5
    and 5; the rule must not accept either neighbour."""
    b = np.array([6.0 * 17 / 16, 6.0 * 19 / 16 * 4, 6.0], np.float32)
    ok, code, recipe = _decide(b, 2688.0)
    assert not ok[0] and not ok[1]
    assert ok[2] and code[2] == recipe[2] == 0x38
    # The recipe rounds those ties to the even significand: 1.0625 -> 1.0
    # (0x38), 4.75 -> 5.0 (0x4A).
    assert recipe[0] == 0x38 and recipe[1] == 0x4A
