"""The multi-rank (data-parallel replica) path of bench.py on CPU ranks.

Two gloo ranks exercise what the N-GPU benchmark relies on without a GPU:
the max-over-ranks reduction of the timed region, the whole-job
throughput formula, per-rank token inputs with shared weights, and the
reference arm doing its work on rank 0 only.
"""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import moe_synth
    cfg = moe_synth.TINY
    # each rank "measures" a different time; the job takes the slowest
    mine = 10.0 + 5.0 * rank
    slowest = bench.max_over_ranks(mine, "cpu")
    value = bench.whole_job_throughput(cfg.T, world, 100, slowest)
    inp = bench.rank_inputs(cfg, rank, world)
    # gather x and W1 checksums from every rank
    sig = torch.tensor([inp["x"].float().sum().item(), inp["w1"].float().sum().item()],
                       dtype=torch.float64)
    sigs = [torch.zeros_like(sig) for _ in range(world)]
    dist.all_gather(sigs, sig)
    # reference arm under torchrun: only rank 0 does work and prints
    args = type("A", (), dict(workload="tiny", warmup=0, steps=1, gpus=world))()
    rc = bench.run_reference(args) if rank != 0 else 0
    torch.save(dict(slowest=slowest, value=value, sigs=[s.tolist() for s in sigs], rc=rc),
               os.path.join(out_dir, f"rank{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    port = 29500 + (os.getpid() % 2000)
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [torch.load(tmp_path / f"rank{r}.pt") for r in range(world)]
    for r in res:
        assert r["slowest"] == 15.0                      # max over ranks, seen by every rank
        assert r["value"] == pytest.approx(2 * 64 * 100 / 0.015)
    sigs = res[0]["sigs"]
    assert sigs[0][0] != sigs[1][0]                      # each replica has its own tokens
    assert sigs[0][1] == sigs[1][1]                      # and the same expert weights
    assert res[1]["rc"] == 0                             # reference arm: rank 1 exits at once


def test_single_process_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_throughput(4096, 1, 10, 20.0) == pytest.approx(4096 * 10 / 0.02)
