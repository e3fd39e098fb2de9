"""The vocabulary-sharded entry points' host side, on the CPU: the shard boundaries, the record slots per row,
and the rank-ordered exchange of the shards' records, run as two gloo ranks ("[WS2][Logprob] Deterministic SM90
linear_logp ...", Tensor parallelism: partials exchanged by an all-gather with no reduction in transit, placed
in rank order). The merge itself runs on the GPU (tests/test_gpu_shard.py)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as tmp

import top_sampling_gb300 as ts

WORLD = 2
B, NP = 3, 5


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("dtype,unit", [(torch.bfloat16, 2048), (torch.float32, 1024)])
def test_piece_aligned_bounds_cover_the_row_in_rank_order(dtype, unit):
    for V, R in [(151936, 2), (151936, 8), (32000, 4), (262144, 8), (5000, 2)]:
        b = ts.shard_bounds(V, R, dtype)
        assert len(b) == R and b[0][0] == 0
        assert all(v0 + n == b[i + 1][0] for i, (v0, n) in enumerate(b[:-1]))      # contiguous, rank order
        assert b[-1][0] + b[-1][1] == V
        assert all(v0 % unit == 0 for v0, _ in b)                                    # on piece boundaries
    b = ts.shard_bounds(151936, 2, dtype, align_to_pieces=False)
    assert all(v0 % (8 if dtype == torch.bfloat16 else 4) == 0 for v0, _ in b)
    with pytest.raises(ValueError):
        ts.shard_bounds(3000, 4, dtype)                                               # fewer pieces than shards


def test_record_slots_are_the_most_pieces_of_any_shard():
    b = ts.shard_bounds(151936, 2, torch.bfloat16)                                    # 38 * 2048 + the rest
    assert ts.shard_record_slots(b, torch.bfloat16) == 38
    assert ts.shard_record_slots(ts.shard_bounds(32000, 4, torch.float32), torch.float32) == 8
    lib = ts.load()
    assert lib.vsamp_shard_pieces(ts.VSAMP_BF16, 2048) == 1 and lib.vsamp_shard_pieces(ts.VSAMP_BF16, 2049) == 2
    assert lib.vsamp_shard_pieces(ts.VSAMP_F32, 1) == 1 and lib.vsamp_shard_pieces(ts.VSAMP_F32, 0) == 0
    assert lib.vsamp_shard_workspace_size(ts.VSAMP_F32, 4, 32000) == 256 + 4 * 32 * 128


def _records(rank):
    """Bytes that name their own (rank, row, slot): what the exchange must put where."""
    r = torch.empty((B, NP, ts.PIECE_REC_BYTES), dtype=torch.uint8)
    for row in range(B):
        for k in range(NP):
            r[row, k, 0], r[row, k, 1], r[row, k, 2] = rank, row, k
            r[row, k, 3:] = (rank * 31 + row * 7 + k) % 251
    w = torch.full((B, ts.SHARD_WIN_BYTES), 100 + rank, dtype=torch.uint8)
    w[:, 1] = torch.arange(B, dtype=torch.uint8)
    return r, w


def _rank_main(rank, port, out_dir):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        recs, win = _records(rank)
        all_r, all_w = ts.gather_shard_records(recs, win)
        torch.save((all_r, all_w), os.path.join(out_dir, f"gathered{rank}.pt"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_gather_records_in_rank_order(tmp_path):
    port = _free_port()
    tmp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=WORLD, join=True, start_method="spawn")
    for rank in range(WORLD):
        all_r, all_w = torch.load(tmp_path / f"gathered{rank}.pt")
        assert tuple(all_r.shape) == (WORLD, B, NP, ts.PIECE_REC_BYTES)
        assert tuple(all_w.shape) == (WORLD, B, ts.SHARD_WIN_BYTES)
        for r in range(WORLD):                 # every rank sees the same [R, B, NP] layout, rank r at index r
            want_r, want_w = _records(r)
            assert torch.equal(all_r[r], want_r) and torch.equal(all_w[r], want_w)
