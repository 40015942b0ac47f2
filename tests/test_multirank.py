"""Replica sharding and the cross-rank timing reduction, as world_size-2 gloo
ranks on the CPU (the bench's N > 1 path without a GPU)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from cached_masked_decoding_gb300 import configs, replicas, synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = configs.TINY
        sh = replicas.shard(rank, world, 3)
        pr = synth.prompts(cfg, 0, sh.batch, 32, first_seq=sh.first_seq)
        dist.barrier()
        elapsed, tokens = replicas.reduce_timing(10.0 + 5.0 * rank, 100 * (rank + 1))
        np.savez(os.path.join(out_dir, f"r{rank}.npz"), prompts=pr, elapsed=elapsed, tokens=tokens,
                 first=sh.first_seq, gb=sh.global_batch)
    finally:
        dist.destroy_process_group()


def test_shard_bounds():
    assert replicas.shard(0, 1, 4).first_seq == 0
    assert replicas.shard(3, 4, 2).first_seq == 6
    assert replicas.shard(1, 2, 5).global_batch == 10
    with pytest.raises(ValueError):
        replicas.shard(2, 2, 1)
    with pytest.raises(ValueError):
        replicas.shard(0, 1, 0)


def test_single_rank_reduce_is_identity():
    assert replicas.reduce_timing(3.5, 7) == (3.5, 7)


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [np.load(tmp_path / f"r{r}.npz") for r in range(world)]
    # every rank sees the max of the elapsed times and the sum of the tokens
    for r in res:
        assert float(r["elapsed"]) == 15.0
        assert int(r["tokens"]) == 300
        assert int(r["gb"]) == 6
    # the shards tile the global batch: rank r's prompts are rows [3r, 3r+3) of
    # the single-process prompt matrix of the whole batch
    whole = synth.prompts(configs.TINY, 0, 6, 32)
    got = np.concatenate([r["prompts"] for r in res])
    np.testing.assert_array_equal(got, whole)
    assert [int(r["first"]) for r in res] == [0, 3]
