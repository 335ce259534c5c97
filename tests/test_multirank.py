"""The multi-GPU launch of bench.py, exercised as world-size-2 gloo ranks on
the CPU: each rank draws its own shard (no data-path collective), the
timing is the max over ranks, the value aggregates all ranks' work, and the
reference arm runs on rank 0 only."""

import os
import socket
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    from separator_token_kv_sep_b300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank time: the max over ranks is what every rank sees
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        cfg = synth.TINY_FWD
        _, _, _, _, ids = synth.prefill_inputs(cfg, seed=bench.shard_seed(cfg.seed, rank))
        shard = bench.visited_pairs_per_head(ids, cfg.a, cfg.n)
        total = bench.max_over_ranks(float(shard), world)  # any rank's shard size
        ids_all = [None] * world
        dist.all_gather_object(ids_all, ids)
        ref = bench.run_reference(type("A", (), {"warmup": 0, "steps": 1})(), rank, world)
        out[rank] = {"t": t, "distinct": not np.array_equal(ids_all[0], ids_all[1]),
                     "shape": ids.shape, "ref_none": ref is None, "total": total}
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(600)
def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0]["t"] == res[1]["t"] == 15.0
    assert res[0]["distinct"] and res[1]["distinct"]
    assert res[0]["shape"] == res[1]["shape"]
    assert res[0]["ref_none"] is False and res[1]["ref_none"] is True


def test_aggregate_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 3 steps x 1e12 FLOP in 1.5 s (the slowest rank) = 4 TFLOP/s
    assert bench.aggregate_value(1e12, 2, 3, 1500.0) == pytest.approx(4.0)
    assert bench.shard_seed(1002, 0) != bench.shard_seed(1002, 1)
