"""Row sharding across ranks: host logic, checked on CPU with gloo (world size 2).

Each rank computes its rows' share of Y with the fp64 oracle (the GPU path is
exercised by the GPU tests), the shares are all-gathered through
torch.distributed, and the result must equal the unsharded oracle exactly:
output rows are independent, so sharding changes no arithmetic.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_weight_only_groupwise_gb300 import sharding, synth


def test_row_shard_covers_and_aligns():
    for N in (1, 15, 16, 17, 129, 5120, 12288):
        for world in (1, 2, 3, 4, 8):
            spans = [sharding.row_shard(N, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c and a <= b
            for a, b in spans[:-1]:
                assert a % 16 == 0 and b % 16 == 0
            widths = [b - a for a, b in spans]
            assert max(widths) - min(widths) <= 16


def _worker(rank, world, port, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    N, K, T = 200, 192, 3
    w = synth.weights(4, N, K, 5)
    x = synth.activations(4, T, K, outliers=True)
    codes, scales, start, stop = sharding.shard_inputs(w["packed"], w["scales"], N, world, rank)
    y_local, _ = oracle.gemm(5, codes, scales, x, stop - start, K)
    y = sharding.gather_columns(torch.from_numpy(y_local), N)
    if rank == 0:
        np.save(result_path, y.numpy())
    dist.destroy_process_group()


def test_gathered_shards_equal_unsharded_oracle(tmp_path):
    import oracle
    world = 2
    port = 29500 + (os.getpid() % 2000)
    out = str(tmp_path / "y.npy")
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    N, K, T = 200, 192, 3
    w = synth.weights(4, N, K, 5)
    x = synth.activations(4, T, K, outliers=True)
    ref, _ = oracle.gemm(5, w["packed"], w["scales"], x, N, K)
    got = np.load(out)
    assert np.array_equal(got, ref)
