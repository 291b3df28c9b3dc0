"""Data parallelism over the batch (one process per GPU): the split, the
shard generator, and a two-rank run over ``gloo`` on the CPU.

Attention rows of different (batch, head) pairs never interact, so a global
batch split into contiguous shards needs no exchange: the ranks' outputs,
put side by side, are the output of the whole batch.  The two-rank test
checks exactly that with the oracle on each rank's shard, and the maximum
over ranks the benchmark takes for its step time."""
import math
import os
import socket

import numpy as np
import pytest

import attn_inputs
import oracle
from exact_attention_forward_10_gb300 import shard


@pytest.mark.parametrize("gb,world", [(2, 1), (4, 2), (5, 3), (16, 8), (3, 4)])
def test_batch_range_covers_each_row_once(gb, world):
    rows = []
    for r in range(world):
        b0, b1 = shard.batch_range(gb, world, r)
        assert 0 <= b0 <= b1 <= gb
        rows += list(range(b0, b1))
    assert rows == list(range(gb))
    sizes = [shard.batch_range(gb, world, r)[1] - shard.batch_range(gb, world, r)[0]
             for r in range(world)]
    assert max(sizes) - min(sizes) <= 1


def test_batch_range_rejects_bad_requests():
    for args in [(4, 0, 0), (4, 2, 2), (4, 2, -1), (-1, 2, 0)]:
        with pytest.raises(ValueError):
            shard.batch_range(*args)


def test_shard_generator_is_a_slice_of_the_global_batch():
    full = attn_inputs.make_qkv(5, 2, 40, 64, "bf16", seed=11)
    for b0, b1 in [(0, 5), (0, 2), (2, 4), (4, 5), (3, 3)]:
        part = attn_inputs.make_qkv_shard(5, b0, b1, 2, 40, 64, "bf16", seed=11)
        for a, b in ((part.q, full.q), (part.k, full.k), (part.v, full.v)):
            np.testing.assert_array_equal(a, b[b0:b1])
    with pytest.raises(ValueError):
        attn_inputs.make_qkv_shard(5, 4, 6, 2, 40, 64, "bf16", seed=11)


def test_max_over_ranks_without_a_group():
    assert shard.max_over_ranks([1.5, 2.0]) == [1.5, 2.0]


GB, H, S, D = 4, 2, 96, 64


def _rank_main(rank, world, port, causal, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import torch
        b0, b1 = shard.batch_range(GB, world, rank)
        x = attn_inputs.make_qkv_shard(GB, b0, b1, H, S, D, "fp16", seed=21)
        o, lse = oracle.attn_fwd(x.q, x.k, x.v, causal, 1 / math.sqrt(D), threads=1)
        # gather the shards (test only: the forward itself exchanges nothing)
        parts_o = [torch.zeros((shard.batch_range(GB, world, r)[1] - shard.batch_range(GB, world, r)[0],
                                H, S, D), dtype=torch.float64) for r in range(world)]
        parts_l = [torch.zeros(p.shape[:3], dtype=torch.float64) for p in parts_o]
        dist.all_gather(parts_o, torch.from_numpy(np.ascontiguousarray(o)))
        dist.all_gather(parts_l, torch.from_numpy(np.ascontiguousarray(lse)))
        # the step time the benchmark keeps: the slowest rank
        slowest = shard.max_over_ranks([1.0 + rank, 10.0 - rank])
        if rank == 0:
            np.save(os.path.join(out_dir, "o.npy"), torch.cat(parts_o).numpy())
            np.save(os.path.join(out_dir, "lse.npy"), torch.cat(parts_l).numpy())
            np.save(os.path.join(out_dir, "slowest.npy"), np.asarray(slowest))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("causal", [False, True])
def test_two_ranks_over_gloo_equal_the_whole_batch(tmp_path, causal):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), causal, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    x = attn_inputs.make_qkv(GB, H, S, D, "fp16", seed=21)
    ro, rl = oracle.attn_fwd(x.q, x.k, x.v, causal, 1 / math.sqrt(D))
    np.testing.assert_array_equal(np.load(tmp_path / "o.npy"), ro)
    np.testing.assert_array_equal(np.load(tmp_path / "lse.npy"), rl)
    assert np.load(tmp_path / "slowest.npy").tolist() == [2.0, 10.0]
