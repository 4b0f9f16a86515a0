"""Host-side logic of bench.py (no GPU): the byte accounting, pinned to the
bandwidths torchao's cast_bench.py printed for the dim1 cast, and the
max-over-ranks timing on a world_size-2 gloo group."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "torchao_dim1_cast_bench.txt")


def golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        mode, M, K, block, t_us, gbps = line.split()
        rows.append((mode, int(M), int(K), int(block), float(t_us), float(gbps)))
    return rows


def test_byte_accounting_matches_printed_bandwidths():
    rows = golden_rows()
    assert len(rows) == 3
    for mode, M, K, block, t_us, gbps in rows:
        assert block == 32
        nbytes = bench.mx_bytes(M, K, rowwise=False, colwise=True)
        assert nbytes == 813_694_976
        assert abs(nbytes / (t_us * 1e-6) / 1e9 - gbps) <= 1e-9 * gbps, mode


def test_byte_accounting_other_workloads():
    assert bench.mx_bytes(16384, 16384) == 1_090_519_040
    assert bench.mx_bytes(8192, 8192, dbias=True) == 272_662_528
    assert bench.mx_bytes(8192, 14336, gated=True) == 711_983_104
    assert bench.mx_bytes(8192, 14336) == 477_102_080
    assert bench.nvfp4_bytes(16384, 8192) == 419_430_408


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(10.0 + rank, world)
    bench.barrier(world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == {0: 11.0, 1: 11.0}


def test_gated_backward_byte_accounting():
    """Gated backward: the [M, 2N] output of a plain cast plus the grad read."""
    for M, N in ((8192, 14336), (64, 96)):
        assert bench.dgated_bytes(M, N) == bench.mx_bytes(M, 2 * N) + 2 * M * N
