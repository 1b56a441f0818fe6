"""The multi-rank path on CPU: two gloo ranks.

The (sequence, head) units are independent, so ranks shard whole sequences
and share nothing on the data path; the only collectives are the timing
aggregation (max of the per-rank times, sum of the units).  These tests run
the oracle as each rank's worker, so they need no GPU.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import gdn_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        inp = gdn_inputs.make_inputs(4321, B=5, T=3, kh=2, vh=6, kd=16, vd=8)
        lo, hi = bench.shard_range(inp.B, world, rank)
        mine = inp.heads(range(lo, hi), range(inp.vh))
        S, o = oracle.run_inputs(mine)
        # gather the shards on every rank (object collective, CPU only)
        got = [None] * world
        dist.all_gather_object(got, (lo, hi, S, o))
        ms, units, rate = bench.aggregate(1.0 + rank, (hi - lo) * inp.vh * 10,
                                          dist, "cpu")
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"),
                 S=np.concatenate([g[2] for g in sorted(got, key=lambda g: g[0])]),
                 o=np.concatenate([g[3] for g in sorted(got, key=lambda g: g[0])]),
                 agg=np.array([ms, units, rate]))
    finally:
        dist.destroy_process_group()


def test_shard_range_covers_everything():
    for n in (0, 1, 5, 64, 97):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_range(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_shard_exactly(tmp_path, oracle_mod):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
             join=True)
    inp = gdn_inputs.make_inputs(4321, B=5, T=3, kh=2, vh=6, kd=16, vd=8)
    S_full, o_full = oracle_mod.run_inputs(inp)
    for r in range(world):
        d = np.load(tmp_path / f"rank{r}.npz")
        assert np.array_equal(d["S"], S_full)
        assert np.array_equal(d["o"], o_full)
        ms, units, rate = d["agg"]
        assert ms == 2.0                      # slowest rank
        assert units == inp.B * inp.vh * 10   # every rank's units
        assert rate == pytest.approx(units / 2e-3)
