"""Seeded synthetic inputs for the quantization workloads.

This module only draws random numbers and rounds them to bf16; it holds none
of the quantization arithmetic.  Both the CUDA-path tests / benchmark and the
oracle checks take their inputs from here, so the two sides see the same bits.

Random numbers come from numpy's Philox counter-based generator, one
independent stream per random component (``SeedSequence.spawn``), drawn in
float32 and rounded once to bf16 with round-to-nearest-even.  Every generator
returns the bf16 bit patterns as a C-contiguous ``numpy.uint16`` array.

Workload recipes (distribution, structure and default sizes):

* ``plain_small``   128x256 N(0,1), seed 0; the 32x32 tile at rows 0-31,
                    cols 0-31 is all zero and the tile at rows 32-63,
                    cols 64-95 is scaled by 2^-130 (bf16 subnormals), so both
                    the rowwise and the colwise blocks there hit the zero and
                    the clamped-scale cases.
* ``rowcol``        16384x16384 N(0,1), seed 5 (the rowwise+colwise cast).
* ``dim1``          16384x16384 N(0,1) times one lognormal(0, 2) factor
                    exp(2 z) per row, seed 1 (the colwise-only cast).
* ``dbias``         8192x8192 N(0,1), seed 2; 0.1% of entries times 1000;
                    1% of the 1x32 row blocks all zero and 1% scaled by
                    2^-130 (zero wins over subnormal wins over outlier).
* ``swiglu``        x[8192, 2*14336] = [gate | up], gate N(0, std 2),
                    up N(0,1), seed 3.
* ``gelu``          8192x14336 N(0,1), seed 3 (its own stream).
* ``nvfp4``         16384x8192 N(0,1), 0.1% of entries times 100, seed 4.
* ``device_normal`` any M x K N(0,1) drawn on a CUDA device with torch's
                    seeded generator (for sizes past 2^31 elements, where a
                    host draw would cost minutes); returned as a bf16 device
                    tensor whose windows are copied back for checking.
"""
import numpy as np

ROW_CHUNK = 1024


def f32_to_bf16_bits(f):
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    b = f.view(np.uint32)
    rounded = (b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits):
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def _streams(seed, n):
    return [np.random.Generator(np.random.Philox(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _normal_rows(gen, M, K, std=1.0, row_factor=None, out=None):
    """Draw an M x K float32 N(0, std^2) matrix and round it to bf16 bits,
    ROW_CHUNK rows at a time to bound host memory."""
    if out is None:
        out = np.empty((M, K), np.uint16)
    for r0 in range(0, M, ROW_CHUNK):
        r1 = min(M, r0 + ROW_CHUNK)
        f = gen.standard_normal((r1 - r0, K), dtype=np.float32)
        if std != 1.0:
            f *= np.float32(std)
        if row_factor is not None:
            f *= row_factor[r0:r1, None]
        out[r0:r1] = f32_to_bf16_bits(f)
    return out


def plain_small(M=128, K=256, seed=0):
    (g,) = _streams(seed, 1)
    f = g.standard_normal((M, K), dtype=np.float32)
    if M >= 32 and K >= 32:
        f[0:32, 0:32] = 0.0
    if M >= 64 and K >= 96:
        f[32:64, 64:96] *= np.float32(2.0 ** -130)
    return f32_to_bf16_bits(f)


def rowcol(M=16384, K=16384, seed=5):
    (g,) = _streams(seed, 1)
    return _normal_rows(g, M, K)


def dim1(M=16384, K=16384, seed=1):
    g_data, g_row = _streams(seed, 2)
    row_factor = np.exp(np.float32(2.0) * g_row.standard_normal(M, dtype=np.float32)).astype(np.float32)
    return _normal_rows(g_data, M, K, row_factor=row_factor)


def dbias(M=8192, K=8192, seed=2):
    g_data, g_out, g_blk = _streams(seed, 3)
    out = np.empty((M, K), np.uint16)
    nb = K // 32
    for r0 in range(0, M, ROW_CHUNK):
        r1 = min(M, r0 + ROW_CHUNK)
        f = g_data.standard_normal((r1 - r0, K), dtype=np.float32)
        outlier = g_out.random((r1 - r0, K)) < 0.001
        f[outlier] *= np.float32(1000.0)
        u = g_blk.random((r1 - r0, nb))
        zero_blk = u < 0.01
        sub_blk = (u >= 0.01) & (u < 0.02)
        fb = f.reshape(r1 - r0, nb, 32)
        fb[sub_blk] *= np.float32(2.0 ** -130)
        fb[zero_blk] = 0.0
        out[r0:r1] = f32_to_bf16_bits(f)
    return out


def swiglu(M=8192, N=14336, seed=3):
    g_gate, g_up = _streams(seed, 2)
    x = np.empty((M, 2 * N), np.uint16)
    _normal_rows(g_gate, M, N, std=2.0, out=x[:, :N])
    _normal_rows(g_up, M, N, out=x[:, N:])
    return x


def gelu(M=8192, K=14336, seed=3):
    g = _streams(seed, 3)[2]
    return _normal_rows(g, M, K)


def nvfp4(M=16384, K=8192, seed=4):
    g_data, g_out = _streams(seed, 2)
    out = np.empty((M, K), np.uint16)
    for r0 in range(0, M, ROW_CHUNK):
        r1 = min(M, r0 + ROW_CHUNK)
        f = g_data.standard_normal((r1 - r0, K), dtype=np.float32)
        f[g_out.random((r1 - r0, K)) < 0.001] *= np.float32(100.0)
        out[r0:r1] = f32_to_bf16_bits(f)
    return out


WORKLOADS = {
    "plain_small": plain_small,
    "rowcol": rowcol,
    "dim1": dim1,
    "dbias": dbias,
    "swiglu": swiglu,
    "gelu": gelu,
    "nvfp4": nvfp4,
}


def device_normal(M, K, seed, device="cuda", chunk_rows=4096):
    """M x K N(0,1) bf16 drawn on `device` (torch's Philox, seeded), rounded
    once from float32 to bf16 (round to nearest even), chunk_rows rows at a
    time."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty((M, K), dtype=torch.bfloat16, device=device)
    for r0 in range(0, M, chunk_rows):
        r1 = min(M, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0, K), generator=g, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
    return out
