"""Row sharding across ranks (the multi-GPU benchmark path), run as two gloo ranks on the CPU.

Rows are independent, so N ranks each sample their own rows with no data-path collective; the Philox
row word is the global row index, which makes every draw independent of how rows are spread over
ranks. The ranks only meet for the barrier around the timed region and the MAX of their times.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench
import workloads
from oracle import sampler as osm

WORLD = 2
ROWS_PER_RANK = 3


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _draw(batch, rows, row_ids, step=0):
    return [osm.sample_row(batch.logits[r], batch.dtype, batch.temperature[r], batch.top_k[r], batch.top_p[r],
                           batch.min_p[r], int(batch.seed[r]), int(g), step).token for r, g in zip(rows, row_ids)]


def _rank_main(rank, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        batch = workloads.c1(B=WORLD * ROWS_PER_RANK)
        gids = bench.shard_row_ids(rank, ROWS_PER_RANK)
        toks = _draw(batch, gids, gids)
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, (rank, gids.tolist(), toks))
        dist.barrier()
        slowest = bench.max_over_ranks(10.0 + rank, dist)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([slowest] + [t for _, _, ts in sorted(gathered) for t in ts], dtype=np.float64))
        with open(os.path.join(out_dir, f"ids{rank}.txt"), "w") as f:
            f.write(" ".join(str(i) for _, ids, _ in sorted(gathered) for i in ids))
    finally:
        dist.destroy_process_group()


def test_shard_row_ids_partition_the_batch():
    ids = np.concatenate([bench.shard_row_ids(r, 5) for r in range(4)])
    assert np.array_equal(ids, np.arange(20))


def test_job_throughput_counts_every_rank():
    assert bench.job_rows_per_s(4, 256, 100, 1000.0) == pytest.approx(4 * 256 * 100)
    assert bench.max_over_ranks(3.5) == 3.5


def test_two_gloo_ranks_match_one_process(tmp_path):
    port = _free_port()
    tmp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=WORLD, join=True, start_method="spawn")
    whole = workloads.c1(B=WORLD * ROWS_PER_RANK)
    rows = list(range(WORLD * ROWS_PER_RANK))
    want = _draw(whole, rows, rows)
    for r in range(WORLD):
        got = np.load(tmp_path / f"rank{r}.npy")
        assert got[0] == 10.0 + (WORLD - 1)                 # MAX over the ranks' times
        assert [int(t) for t in got[1:]] == want            # sharded draws == unsharded draws
        ids = [int(i) for i in (tmp_path / f"ids{r}.txt").read_text().split()]
        assert ids == rows
