"""The N>1 host logic of bench.py, on CPU with the gloo backend (world size 2).

The path shards by batch with no data exchange: each rank draws its own
batch (different seed, same shapes) and the only collective is the max of
the timed region over ranks.  These tests run that logic in two processes.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import bench
    import workloads

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        elapsed = 10.0 + 5.0 * rank            # pretend rank 1 was slower
        m = bench.max_over_ranks(elapsed, dist)
        case = bench._make_rank_case("spec_verify_b16_t8_bf16", rank)
        base = workloads.make_config("spec_verify_b16_t8_bf16")
        np.save(os.path.join(out_dir, f"k{rank}.npy"), case.k)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{m} {case.B} {case.T} {int(np.array_equal(case.k, base.k))}\n")
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_and_timing(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0 = open(tmp_path / "r0.txt").read().split()
    r1 = open(tmp_path / "r1.txt").read().split()
    # both ranks see the max over ranks
    assert float(r0[0]) == 15.0 and float(r1[0]) == 15.0
    # same shapes on every rank (weak scaling: per-rank work is fixed)
    assert r0[1:3] == r1[1:3] == ["16", "8"]
    # rank 0 is the named workload itself; rank 1 is an independent batch
    assert r0[3] == "1" and r1[3] == "0"
    k0, k1 = np.load(tmp_path / "k0.npy"), np.load(tmp_path / "k1.npy")
    assert k0.shape == k1.shape and not np.array_equal(k0, k1)


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.rank_seed(1003, 0) == 1003
    assert len({bench.rank_seed(1003, r) for r in range(8)}) == 8


def test_bench_arguments():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.config == "rollback_b128_t16_bf16"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def test_algorithmic_bytes_rollback():
    import bench
    import workloads
    case = workloads.make_config("rollback_b128_t16_bf16")
    rec, rep = bench.algorithmic_bytes(case, case.accepted)
    state = 128 * 32 * 128 * 128 * 4
    act = int(case.mask.sum())
    assert rec == 2 * state + act * (2 * 16 * 128 + 32 * 128 + 2 * 32 + 2 * 32 * 128
                                     + 32 * 128 + 32) * 2 + 128 * 16 * 4
    act11 = int(case.mask[:, :11].sum())
    assert rep == 2 * state + act11 * (32 * 128 + 32 * 128 + 32) * 2 + 128 * 11 * 4
