"""The row-sharded exchange (NVFP4 amax all-reduce MAX, dbias all-reduce
SUM) on a world_size-2 gloo group on the CPU, with the oracle standing in
for each rank's kernels; every rank's outputs are checked against the
oracle run over the whole matrix in one process."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth

from fp4_quantization_gb300 import sharded  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_amax(panel_bits):
    return torch.tensor([oracle.bf16_amax(panel_bits)], dtype=torch.float32)


def _oracle_nvfp4(panel_bits, flags, amax):
    return oracle.nvfp4_quantize(panel_bits, tensor_amax=float(amax[0]), flags=flags)


def _oracle_mx(panel_bits, flags):
    out = oracle.mx_quantize(panel_bits, flags)
    out["dbias"] = torch.from_numpy(out["dbias"])
    return out


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # NVFP4: the tensor amax is planted in rank 1's panel, so rank 0's
        # own amax is smaller and only the all-reduce gives it the right G.
        x = synth.nvfp4(M=256, K=128, seed=21)
        x[200, 5] = synth.f32_to_bf16_bits(np.array([3000.0], np.float32))[0]
        m0, m1 = sharded.row_panel(256, rank, world)
        out = sharded.nvfp4_quantize_transpose_sharded(
            x[m0:m1], 3, quantize=_oracle_nvfp4, amax_fn=_oracle_amax)
        full = oracle.nvfp4_quantize(x, flags=3)
        nv_ok = (np.array_equal(out["q_row"], full["q_row"][m0:m1])
                 and np.array_equal(out["s_row"], full["s_row"][m0:m1])
                 and np.array_equal(out["q_t"], full["q_t"][:, m0 // 2:m1 // 2])
                 and np.array_equal(out["s_t"], full["s_t"][:, m0 // 16:m1 // 16])
                 and out["global_scale"] == full["global_scale"])
        # dbias: the all-reduced panel sums against the whole-matrix sums.
        y = synth.dbias(M=320, K=96, seed=22)
        m0, m1 = sharded.row_panel(320, rank, world)
        out = sharded.mx_quantize_rowcol_dbias_sharded(y[m0:m1], 3, quantize=_oracle_mx)
        full = oracle.mx_quantize(y, 3 | oracle.DBIAS)
        tol = 1e-6 * np.abs(synth.bf16_bits_to_f32(y).astype(np.float64)).sum(axis=0) + 1e-30
        err = np.abs(out["dbias"].numpy().astype(np.float64) - full["dbias"].astype(np.float64))
        db_ok = bool(np.all(err <= tol)) and np.array_equal(out["q_col"], full["q_col"][:, m0:m1])
        results[rank] = (nv_ok, db_ok)
    finally:
        dist.destroy_process_group()


def test_sharded_exchange_gloo_world2():
    world = 2
    with mp.get_context("spawn").Manager() as manager:
        results = manager.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        assert dict(results) == {0: (True, True), 1: (True, True)}


def test_row_panels_cover_the_rows_in_whole_blocks():
    for M, world in ((256, 2), (320, 3), (96, 4), (32, 2)):
        spans = [sharded.row_panel(M, r, world) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == M
        for (a0, a1), (b0, _) in zip(spans, spans[1:]):
            assert a1 == b0 and a0 % 32 == 0
