"""World-size-2 gloo test of the multi-rank host logic (no GPU).

Each rank takes its share of a packed varlen batch (sharded by sequence, no exchange on
the data path), runs it, and the gathered per-sequence results must equal the unsharded
run exactly.  The fp64 oracle stands in for the device compute here; the property under
test is the sharding and gathering, plus the max-over-ranks timing reduction.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from gated_deltanet_linear_11_gb300 import inputs
from gated_deltanet_linear_11_gb300.shard import max_over_ranks, partition_sequences, sub_batch

LENS = [5, 70, 1, 33, 128, 12, 64]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = inputs.scan_inputs(81, LENS, 1, 2, 16, 8, dtype=torch.float32,
                               init_state_std=0.1)
        parts = partition_sequences(LENS, world)
        mine = parts[rank]
        tok, cu_sub = sub_batch(x["cu_seqlens"].numpy(), mine)
        tok_t = torch.from_numpy(tok)
        o, hT = oracle.gated_delta_rule(x["q"][tok_t], x["k"][tok_t], x["v"][tok_t],
                                        x["g"][tok_t], x["beta"][tok_t], cu_sub,
                                        initial_state=x["initial_state"][mine], nthreads=1)
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, tok, o, hT))
        worst = max_over_ranks(1.0 + rank)
        if rank == 0:
            np.savez(os.path.join(out_dir, "res.npz"), worst=worst,
                     payload=np.array(gathered, dtype=object))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_matches_unsharded(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = np.load(tmp_path / "res.npz", allow_pickle=True)
    assert float(res["worst"]) == 2.0
    x = inputs.scan_inputs(81, LENS, 1, 2, 16, 8, dtype=torch.float32, init_state_std=0.1)
    o_ref, h_ref = oracle.gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                           x["cu_seqlens"], initial_state=x["initial_state"],
                                           nthreads=1)
    seen = set()
    for mine, tok, o, hT in res["payload"]:
        np.testing.assert_array_equal(o, o_ref[tok])
        np.testing.assert_array_equal(hT, h_ref[mine])
        seen |= set(mine)
    assert seen == set(range(len(LENS)))


def test_partition_is_balanced_and_deterministic():
    parts = partition_sequences([100, 1, 50, 50, 3], 2)
    assert parts == partition_sequences([100, 1, 50, 50, 3], 2)
    loads = [sum([100, 1, 50, 50, 3][i] for i in p) for p in parts]
    assert max(loads) - min(loads) <= 3
    assert sorted(i for p in parts for i in p) == list(range(5))
