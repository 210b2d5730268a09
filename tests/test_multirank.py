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


def test_bench_launches_its_own_ranks():
    """``bench.py --gpus 2`` started without a launcher starts two ranks
    itself (torch.distributed.run on 127.0.0.1); the dry-run leg makes no
    CUDA call, so the launcher, the gloo barrier and the max-over-ranks
    timing run here on the CPU.  Rank 0 alone prints one line naming both."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry-run",
                          "--steps", "5", "--warmup", "3"], capture_output=True, text=True, timeout=300,
                         env=env, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(x) for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = lines[0]
    assert line["n_gpus"] == 2 and line["dry_run"] and line["steps"] == 5
    # whole-job rate: both ranks' units over the slowest rank's time
    assert abs(line["value"] - 2 * 1000.0 * 5 / (line["ms_per_step"] * 5 / 1e3)) <= 1e-6 * line["value"]
