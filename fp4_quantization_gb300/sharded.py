"""Row-sharded quantization over the ranks of a torch.distributed group.

Each rank holds a panel of the matrix's rows (a multiple of 32 rows) and
quantizes it on its own GPU.  No MXFP8 or NVFP4 block crosses a panel
boundary, so the codes and scales need no exchange; two quantities do:

* the NVFP4 tensor amax, which every rank needs before it quantizes: one
  all-reduce (MAX) of a single fp32 value;
* the MXFP8 dbias, the column sums over all rows: one all-reduce (SUM) of K
  fp32 values after the quantization (the rank partials are added in the
  collective's order).

Rank r's outputs are its panel's: rowwise codes and scales for its rows, and
the columns [m0, m0 + rows) of the colwise / transposed outputs (their
[K][M] layout puts a rank's rows in a column slice).  The quantize and amax
callables default to this package's CUDA entry points; they are parameters
so that the exchange logic can be exercised without a GPU.
"""
import torch
import torch.distributed as dist

from . import (COLWISE, DBIAS, ROWWISE, bf16_amax, mx_quantize_rowcol,
               nvfp4_quantize_transpose)


def nvfp4_quantize_transpose_sharded(x_panel, flags=ROWWISE | COLWISE, *, group=None,
                                     quantize=None, amax_fn=None):
    """NVFP4 of this rank's row panel with the tensor amax of the whole
    matrix: local amax, all-reduce MAX, then the quantization with that
    amax (so every rank uses the same global scale)."""
    quantize = quantize or nvfp4_quantize_transpose
    amax_fn = amax_fn or bf16_amax
    amax = amax_fn(x_panel)
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return quantize(x_panel, flags, amax=amax)


def mx_quantize_rowcol_dbias_sharded(x_panel, flags=ROWWISE | COLWISE, *, group=None,
                                     quantize=None):
    """MXFP8 of this rank's row panel with dbias over the whole matrix: the
    panel's column sums, then an all-reduce SUM."""
    quantize = quantize or mx_quantize_rowcol
    out = quantize(x_panel, flags | DBIAS)
    dist.all_reduce(out["dbias"], op=dist.ReduceOp.SUM, group=group)
    return out


def row_panel(M, rank, world, multiple=32):
    """[m0, m1) of rank's row panel: M split into `world` panels of whole
    `multiple`-row groups (the last ranks may get one group less)."""
    groups = M // multiple
    per, extra = divmod(groups, world)
    g0 = rank * per + min(rank, extra)
    g1 = g0 + per + (1 if rank < extra else 0)
    return g0 * multiple, g1 * multiple
