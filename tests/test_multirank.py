"""The N > 1 path on CPU: two gloo ranks.

bench.py runs one replica per GPU (weak scaling; sequences of a batch are
independent and carry their own memory, so no data-path collective).  The only
collectives are the timing barrier and the max-over-ranks reduction; this test
runs them with gloo, world size 2, and checks that sharding the batch across
ranks and concatenating reproduces the unsharded result (the oracle on each
rank's batch slice).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import oracle
    from transformer_xl_relative_rel_gb300 import inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    # timing reduction: the slowest rank's time decides
    local = [0.5, 2.0][rank]
    assert bench.max_over_ranks(local, world) == 2.0
    rate = bench.aggregate_rate(100.0, local, world)      # 100 units per rank
    assert abs(rate - 200.0 / 2.0) < 1e-12
    bench.barrier(world)
    # batch sharding: rank r takes sequences [r*B/2, (r+1)*B/2)
    shape = inputs.LayerShape(4, 2, 8, 6, 5)
    p = inputs.unit_layer(shape, 17)
    lo, hi = rank * 2, rank * 2 + 2
    part = oracle.rel_attn(p["q"][:, lo:hi], p["k"][:, lo:hi], p["v"][:, lo:hi], p["r"], p["u"],
                           p["w"], mem_len=shape.mem_len)
    np.save(os.path.join(outdir, f"part{rank}.npy"), part)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_ranks_gloo(tmp_path):
    import oracle
    from transformer_xl_relative_rel_gb300 import inputs
    oracle.build()
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    shape = inputs.LayerShape(4, 2, 8, 6, 5)
    p = inputs.unit_layer(shape, 17)
    full = oracle.rel_attn(p["q"], p["k"], p["v"], p["r"], p["u"], p["w"], mem_len=shape.mem_len)
    parts = np.concatenate([np.load(tmp_path / f"part{r}.npy") for r in range(world)], axis=1)
    assert np.array_equal(parts, full)
