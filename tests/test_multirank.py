"""Multi-rank host logic on CPU (gloo, world size 2).

The path runs as independent replicas: each rank verifies its own requests
and the only collective is the max over ranks of the timed region.  These
tests check that reduction, the whole-job rate, that replicas draw distinct
inputs, and that splitting a batch's requests across ranks (with global
request indices for the Philox counters) reproduces the unsplit batch.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(WORLD),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        world, r, local = bench.dist_env()
        assert (world, r, local) == (WORLD, rank, rank)
        # timings: the slowest rank decides, the rate counts every rank's rounds
        local_ms = 100.0 + 25.0 * rank
        total = bench.max_over_ranks(local_ms, world, "cpu")
        assert total == 125.0
        assert bench.whole_job_rate(world, 50, total) == pytest.approx(2 * 50 / 0.125)
        # a batch of 6 requests split 3 + 3; each rank verifies its share with
        # global request indices
        from speculative_decoding_verification_draft_gb300 import workloads as wl
        full = wl.zipf_batch(6, 3, 257, dtype=torch.float32, temperature=0.9, seed=77)
        tgt, dft = full.numpy_logits()
        tok = full.draft_tokens.numpy()
        ids = np.arange(3 * rank, 3 * rank + 3)
        res = oracle.load().verify_batch(tgt[ids], dft[ids], tok[ids], 0.9, 1234, req_ids=ids)
        mine = torch.from_numpy(np.concatenate([res["n_accepted"][:, None], res["out_tokens"]], 1).astype(np.int64))
        gathered = [torch.empty_like(mine) for _ in range(WORLD)]
        dist.all_gather(gathered, mine)
        if rank == 0:
            torch.save(torch.cat(gathered), os.path.join(out_dir, "sharded.pt"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def sharded(tmp_path_factory):
    out = tmp_path_factory.mktemp("mr")
    mp.start_processes(_rank_main, args=(_free_port(), str(out)), nprocs=WORLD, join=True, start_method="spawn")
    return torch.load(os.path.join(out, "sharded.pt"))


def test_sharded_requests_match_the_unsplit_batch(sharded):
    from speculative_decoding_verification_draft_gb300 import workloads as wl
    full = wl.zipf_batch(6, 3, 257, dtype=torch.float32, temperature=0.9, seed=77)
    tgt, dft = full.numpy_logits()
    ref = oracle.load().verify_batch(tgt, dft, full.draft_tokens.numpy(), 0.9, 1234)
    want = np.concatenate([ref["n_accepted"][:, None], ref["out_tokens"]], 1)
    assert np.array_equal(sharded.numpy(), want)


def test_replicas_draw_distinct_inputs():
    seeds = {bench.replica_seed(r, s) for r in range(8) for s in range(bench.N_SETS)}
    assert len(seeds) == 8 * bench.N_SETS
    assert bench.replica_seed(0, 0) == 2  # one GPU keeps the published workload seed


def test_single_rank_needs_no_collective():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(1, 10, 1000.0) == pytest.approx(10.0)
