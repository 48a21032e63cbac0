"""The multi-rank path on CPU: two gloo ranks (no GPU).

Attention shards by (batch, head) with no exchange step. These tests check the
host logic that does it: the head blocks cover every head once, results
computed rank by rank on those blocks and gathered equal the unsharded
results bit for bit (the oracle stands in for the kernels, which need a GPU),
and the timing's maximum over ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from exact_attention_97_gb300.inputs import make_qkv_do
from exact_attention_97_gb300.shard import head_range, local_heads, max_over_ranks


def test_head_range_covers_each_head_once():
    for n in (0, 1, 7, 64, 256, 1000):
        for world in (1, 2, 3, 8):
            seen = []
            sizes = []
            for r in range(world):
                lo, hi = head_range(n, r, world)
                seen += list(range(lo, hi))
                sizes.append(hi - lo)
            assert seen == list(range(n))
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        head_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, dO = make_qkv_do(2, 3, 40, 8, seed=21, dtype=torch.float32)
        mine = [local_heads(t, rank, world) for t in (q, k, v, dO)]
        o, lse = oracle.attention_fwd(*mine[:3], 0.35, True)
        dq, dk, dv = oracle.attention_bwd(*mine, 0.35, True)
        parts = [None] * world
        dist.all_gather_object(parts, (o, lse, dq, dk, dv))
        peak = max_over_ranks(1.5 + rank)
        if rank == 0:
            full = [np.concatenate([p[i][0] for p in parts], axis=0) for i in range(5)]
            np.savez(out_path, *full, peak=np.array(peak))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_heads_and_agree(tmp_path):
    out = str(tmp_path / "gathered.npz")
    torch.multiprocessing.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                                          start_method="spawn")
    got = np.load(out)
    q, k, v, dO = make_qkv_do(2, 3, 40, 8, seed=21, dtype=torch.float32)
    o, lse = oracle.attention_fwd(q, k, v, 0.35, True)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, 0.35, True)
    for i, ref in enumerate((o, lse, dq, dk, dv)):
        assert np.array_equal(got[f"arr_{i}"], ref.reshape(6, *ref.shape[2:]))
    assert float(got["peak"]) == 2.5


def test_max_over_ranks_without_a_group_is_the_value():
    assert max_over_ranks(3.25) == 3.25
