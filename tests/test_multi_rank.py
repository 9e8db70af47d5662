"""The bench's multi-rank path on CPU: two gloo ranks (no GPU).

`bench.py --gpus N` runs one replica of the decode per rank (the path partitions into
independent sequences, so ranks share nothing on the data path) and reports the whole job:
the maximum of the ranks' times and the sum of their bytes, after a barrier.  These tests
run that aggregation and barrier with world_size 2 over gloo, check that each rank draws its
own batch, and that the reference arm does its work on rank 0 only.
"""
import argparse
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group(backend="gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        bench.barrier()
        # rank k "took" 1.5 + k seconds for 1000 (k + 1) bytes
        sec, nbytes = bench.aggregate(1.5 + rank, 1000 * (rank + 1))
        bench.barrier()
        # the inputs a rank decodes: seed offset by the rank, as run_ours draws them
        wl = W.reduced(W.GQA_B32, 3, 100, 400)
        inp = W.make_inputs(wl, W.SEEDS[0] + rank)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{sec} {nbytes} {int(inp['context_lens'].sum())} "
                    f"{float(inp['q'].float().sum()):.6f}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_bytes(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    lines = [open(tmp_path / f"rank{k}.txt").read().split() for k in range(2)]
    for sec, nbytes, _, _ in lines:
        assert float(sec) == 2.5  # max over ranks
        assert int(nbytes) == 3000  # sum over ranks
    # each rank decodes its own batch (weak scaling: the work per rank is fixed)
    assert (lines[0][2], lines[0][3]) != (lines[1][2], lines[1][3])


def test_aggregate_without_a_process_group_is_the_identity():
    assert not dist.is_initialized()
    assert bench.aggregate(0.25, 1234) == (0.25, 1234)
    bench.barrier()  # no-op


def test_reference_arm_works_on_rank_zero_only():
    args = argparse.Namespace(workload=W.BENCH.name, steps=1, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None


def test_bench_rejects_fewer_than_three_warmup_steps():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--impl", "reference"])
