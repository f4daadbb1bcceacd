"""The multi-rank path on CPU: weak scaling by batch shards, no data-path collective.

Samples are independent through the whole block (LayerNorm per row, the FFN per
sample row, pooling per sample), so N ranks each run the full model on their
own shard of the batch; the only collective is the max over ranks of the timed
region.  These tests cover the host logic that bench.py runs under torchrun:
the batch split, the shard-wise input generator, the max-over-ranks timing and
the whole-job rate, with two gloo ranks on 127.0.0.1.  The per-rank compute is
the oracle on the rank's shard (the CUDA library needs a GPU).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from rankmixer_feature_interaction_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("global_batch,world", [(7, 2), (8, 2), (4096 * 8, 8), (5, 8), (1, 1), (130, 3)])
def test_shard_batch_partitions_the_batch(global_batch, world):
    bounds = [bench.shard_batch(global_batch, world, r) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == global_batch
    for (a0, a1), (b0, b1) in zip(bounds, bounds[1:]):
        assert a1 == b0                                     # contiguous, no overlap, no gap
    sizes = [b - a for a, b in bounds]
    assert max(sizes) - min(sizes) <= 1                     # balanced
    assert sizes == sorted(sizes, reverse=True)             # the first ranks take the remainder


def test_input_shards_concatenate_to_the_global_batch():
    T, D, gb = 3, 10, 2 * synth.SHARD_BLOCK + 9
    whole = synth.make_input_shard(gb, 0, gb, T, D, 11, "f32")
    assert whole.shape == (gb, T, D)
    for world in (1, 2, 3, 5):
        parts = [synth.make_input_shard(gb, *bench.shard_batch(gb, world, r), T, D, 11, "f32") for r in range(world)]
        assert torch.equal(torch.cat(parts, 0), whole)
    assert synth.make_input_shard(gb, 4, 4, T, D, 11, "f32").shape == (0, T, D)
    assert not torch.equal(whole, synth.make_input_shard(gb, 0, gb, T, D, 12, "f32"))
    with pytest.raises(ValueError):
        synth.make_input_shard(gb, 5, gb + 1, T, D, 11, "f32")


def test_job_rate_and_single_process_max():
    assert bench.job_rate(4096, 8, 100, 2.0) == 8 * 4096 * 100 / 2.0
    assert bench.max_over_ranks(3.5) == 3.5                 # no process group: identity


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    import torch.distributed as dist

    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = synth.CONFIGS["tiny_fp32"]
        T, D, k, L = c["T"], c["D"], c["k"], 2
        global_B = 2 * synth.SHARD_BLOCK + 3            # ragged: shards straddle generator blocks
        start, stop = bench.shard_batch(global_B, world, rank)
        layers = synth.to_f64(synth.make_stack(T, D, k, L, 5, "f32", "cpu"))
        X = synth.to_f64(synth.make_input_shard(global_B, start, stop, T, D, 20260101, "f32"))
        oracle.set_num_threads(1)
        pooled = oracle.stack_forward(X, layers)
        # each rank reports its own time; every rank must get the largest
        t_rank = 1.0 + 2.0 * rank
        t_max = bench.max_over_ranks(t_rank)
        gathered = [None] * world
        dist.all_gather_object(gathered, (start, stop, pooled))
        np.save(os.path.join(out_dir, f"rank{rank}_tmax.npy"), np.array([t_max]))
        if rank == 0:
            full = np.concatenate([g[2] for g in sorted(gathered, key=lambda g: g[0])], 0)
            np.save(os.path.join(out_dir, "pooled_sharded.npy"), full)
            np.save(os.path.join(out_dir, "bounds.npy"), np.array([g[:2] for g in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_the_batch_and_take_the_max_time(tmp_path):
    import oracle

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        assert np.load(tmp_path / f"rank{r}_tmax.npy")[0] == 1.0 + 2.0 * (world - 1)
    bounds = np.load(tmp_path / "bounds.npy")
    global_B = 2 * synth.SHARD_BLOCK + 3
    assert bounds.tolist() == [list(bench.shard_batch(global_B, world, r)) for r in range(world)]
    # the ranks' shards, each run on its own, give the single-process result on the whole batch
    c = synth.CONFIGS["tiny_fp32"]
    T, D, k = c["T"], c["D"], c["k"]
    layers = synth.to_f64(synth.make_stack(T, D, k, 2, 5, "f32", "cpu"))
    X = synth.to_f64(synth.make_input_shard(global_B, 0, global_B, T, D, 20260101, "f32"))
    whole = oracle.stack_forward(X, layers)
    sharded = np.load(tmp_path / "pooled_sharded.npy")
    assert sharded.shape == whole.shape
    assert np.array_equal(sharded, whole)


def _train_rank_main(rank: int, world: int, port: int, out_dir: str):
    """Data-parallel training on gloo ranks: each rank's oracle gradients on its shard,
    summed over the ranks by bench.allreduce_grads."""
    import torch.distributed as dist

    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T, D, k, L = 2, 4, 2, 2
        global_B = 2 * synth.SHARD_BLOCK + 3
        start, stop = bench.shard_batch(global_B, world, rank)
        layers = synth.to_f64(synth.make_stack(T, D, k, L, 6, "f32", "cpu"))
        X = synth.to_f64(synth.make_input_shard(global_B, start, stop, T, D, 20260101, "f32"))
        dP = np.random.default_rng(7).standard_normal((global_B, D))[start:stop] / global_B
        oracle.set_num_threads(1)
        _, grads = oracle.stack_backward(X, dP, layers)
        flat = torch.from_numpy(np.concatenate([g[key].reshape(-1) for g in grads for key in oracle.GRAD_KEYS]))
        bench.allreduce_grads(flat)
        if rank == 0:
            np.save(os.path.join(out_dir, "grads_allreduced.npy"), flat.numpy())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_all_reduce_their_shard_gradients(tmp_path):
    """The sum over ranks of the shard gradients is the whole batch's gradient ("RankMixer 详解（1）"
    section 5.2: batch gradients add up over samples), so a replica step needs exactly this one
    exchange."""
    import oracle

    world = 2
    mp.start_processes(_train_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    T, D, k, L = 2, 4, 2, 2
    global_B = 2 * synth.SHARD_BLOCK + 3
    layers = synth.to_f64(synth.make_stack(T, D, k, L, 6, "f32", "cpu"))
    X = synth.to_f64(synth.make_input_shard(global_B, 0, global_B, T, D, 20260101, "f32"))
    dP = np.random.default_rng(7).standard_normal((global_B, D)) / global_B
    _, grads = oracle.stack_backward(X, dP, layers)
    whole = np.concatenate([g[key].reshape(-1) for g in grads for key in oracle.GRAD_KEYS])
    summed = np.load(tmp_path / "grads_allreduced.npy")
    np.testing.assert_allclose(summed, whole, rtol=1e-11, atol=1e-13)
    # without a process group the call leaves the buffer alone
    t = torch.ones(3, dtype=torch.float64)
    bench.allreduce_grads(t)
    assert torch.equal(t, torch.ones(3, dtype=torch.float64))
