"""Whole-matrix oracle outputs at the workload sizes, computed in row panels
on every host core.

MXFP8 and NVFP4 blocks never cross a panel boundary when panels are whole
multiples of 32 rows, so the oracle run panel by panel gives exactly the
oracle's full-matrix output: rowwise outputs are the panels' rows stacked,
colwise (transposed) outputs the panels' columns side by side.  The oracle
calls go through ctypes, which releases the GIL, so a thread pool runs them
in parallel.  Test infrastructure only."""
import concurrent.futures
import os

import numpy as np

# Output key -> (axis the panel's rows run along, output units per input row).
# Colwise outputs are [K][M...]: the panel's rows are its columns.
_MX_LAYOUT = {"q_row": (0, 1), "s_row": (0, 1), "q_col": (1, 1), "s_col": (1, 1 / 32)}
_NV_LAYOUT = {"q_row": (0, 1), "s_row": (0, 1), "q_t": (1, 1 / 2), "s_t": (1, 1 / 16)}


def host_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def run_panels(fn, M, layout, panel_rows=None):
    """fn(r0, r1) returns the oracle's outputs for rows r0..r1 (a dict of
    arrays); returns the full outputs, assembled per `layout`."""
    threads = host_threads()
    if panel_rows is None:
        panel_rows = max(32, (M // (4 * threads)) // 32 * 32)
    bounds = [(r, min(M, r + panel_rows)) for r in range(0, M, panel_rows)]
    full = {}

    def place(part, r0, r1):
        for key, arr in part.items():
            if key in layout:
                axis, per_row = layout[key]
                lo, hi = int(r0 * per_row), int(r1 * per_row)
                if axis == 0:
                    full[key][lo:hi] = arr
                else:
                    full[key][:, lo:hi] = arr

    # The first panel, run alone, gives the outputs' shapes and dtypes.
    first = fn(*bounds[0])
    for key, arr in first.items():
        if key in layout:
            axis, per_row = layout[key]
            shape = list(arr.shape)
            shape[axis] = int(M * per_row)
            full[key] = np.empty(shape, arr.dtype)
    place(first, *bounds[0])
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        list(pool.map(lambda b: place(fn(*b), *b), bounds[1:]))
    return full


def mx_panels(fn, M):
    return run_panels(fn, M, _MX_LAYOUT)


def nvfp4_panels(fn, M):
    return run_panels(fn, M, _NV_LAYOUT)
