"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2).

The path shards by independent (sequence, kv head) units, so the only cross-rank
steps are the seeding of each rank's batch and the max-over-ranks timing; both
run here without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from exact_causal_gqa_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + rank, "cpu")
        prob = inputs.make_config(2, seed=bench.rank_seed(2, rank), B=2)
        checksum = float(prob.q.float().sum())
        sig = [prob.q.shape, prob.k_pages.shape[1:], prob.page_table.shape[1]]
        gathered = [None] * world
        torch.distributed.all_gather_object(gathered, (ms, checksum, sig,
                                                       prob.seq_lens.tolist()))
        if rank == 0:
            out.put(gathered)
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_share_the_slowest_time_and_draw_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    result = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (ms0, sum0, sig0, lens0), (ms1, sum1, sig1, lens1) = result
    assert ms0 == ms1 == 2.0                 # every rank reports the slowest rank
    assert sig0 == sig1                      # same workload shape on every rank
    assert sum0 != sum1 or lens0 != lens1    # but an independent batch per rank


def test_job_rate_counts_all_ranks_units():
    # 2 ranks x 2 GB of KV each in 1 ms (slowest rank) -> 4000 GB/s
    assert bench.job_rate(2e9, 2, 1.0, 1e9) == pytest.approx(4000.0)
    assert bench.rank_seed(2, 0) != bench.rank_seed(2, 1)
