"""The multi-rank path on CPU: two gloo ranks driving the benchmark's own
multi-rank helpers.

The (sequence, head) units are independent, so every rank decodes a batch of
its own (bench.rank_workload) and the data path has no collective; the only
collectives are the timing aggregation (bench.aggregate: the slowest rank's
time, the units of all ranks).  Each rank's worker here is the oracle, so the
test needs no GPU.
"""

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import gdn_inputs

SMALL = dict(B=3, T=2, kh=2, vh=6, kd=16, vd=8)


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
        inp = bench.rank_workload(rank, **SMALL)
        S, o = oracle.run_inputs(inp)
        units = inp.B * inp.vh * inp.T
        ms, total, rate = bench.aggregate(1.0 + rank, units, dist, "cpu")
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), S=S, o=o,
                 q=inp.q, agg=np.array([ms, total, rate]))
    finally:
        dist.destroy_process_group()


def test_rank_batches_are_the_headline_workload_and_distinct():
    r0 = bench.rank_workload(0, **SMALL)
    ref = gdn_inputs.make_workload("decode_b64", **SMALL)
    assert np.array_equal(r0.S, ref.S) and np.array_equal(r0.q, ref.q)
    r1 = bench.rank_workload(1, **SMALL)
    assert r1.S.shape == r0.S.shape and not np.array_equal(r1.S, r0.S)
    assert bench.rank_workload(0).B == 64


def test_two_gloo_ranks(tmp_path, oracle_mod):
    """Each rank's result is exactly that of its own batch computed alone
    (no coupling between ranks), and the aggregate is the slowest rank's
    time with every rank's units."""
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
             join=True)
    for r in range(world):
        d = np.load(tmp_path / f"rank{r}.npz")
        alone = bench.rank_workload(r, **SMALL)
        S_ref, o_ref = oracle_mod.run_inputs(alone)
        assert np.array_equal(d["q"], alone.q)
        assert np.array_equal(d["S"], S_ref)
        assert np.array_equal(d["o"], o_ref)
        ms, units, rate = d["agg"]
        assert ms == 2.0                                  # slowest rank
        assert units == world * SMALL["B"] * SMALL["vh"] * SMALL["T"]
        assert rate == pytest.approx(units / 2e-3)
