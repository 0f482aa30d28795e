"""The bench's N-GPU path on CPU: two `gloo` ranks (spawned processes) run
the host logic that `python -m torch.distributed.run ... bench.py --gpus N`
uses -- rank discovery from the environment, identical seeded replicas of
the workload on every rank, the max-over-ranks reduction of the per-rank
times and the whole-job (weak-scaling) throughput -- without a GPU.  The
path has no exchange step, so the only collective is that reduction."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads as W
        r, lr, ws = bench.dist_env()
        # per-rank times (ms) that differ between ranks: the report is the slowest
        mine = [1.0 + rank, 5.0 - rank, 2.5, 0.25 * (rank + 1)]
        slowest = bench.max_over_ranks(dist, torch.device("cpu"), mine)
        w = W.make("canonical")
        step_bytes = w.append_bytes_int8() + w.decode_bytes_int8()
        value = bench.job_throughput(ws, step_bytes, slowest[0])
        out.put({"rank": r, "local_rank": lr, "world": ws, "slowest": slowest, "value": value,
                 "step_bytes": step_bytes, "lens": w.context_lens.tolist()})
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_replicate():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in res] == [0, 1] and all(d["world"] == world for d in res)
    assert [d["local_rank"] for d in res] == [0, 1]
    for d in res:
        # max over ranks, element by element, the same on every rank
        assert d["slowest"] == [2.0, 5.0, 2.5, 0.5]
    # replicas: every rank builds the same seeded workload
    assert res[0]["lens"] == res[1]["lens"] and res[0]["step_bytes"] == res[1]["step_bytes"]
    # weak scaling: N replicas' bytes over the slowest rank's step time
    expect = world * res[0]["step_bytes"] / (2.0e-3) / 1e9
    assert all(np.isclose(d["value"], expect, rtol=1e-12) for d in res)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(None, None, [3, 1.5]) == [3.0, 1.5]
    assert np.isclose(bench.job_throughput(1, 2e9, 1.0), 2000.0)
    assert np.isclose(bench.job_throughput(4, 2e9, 2.0), 4000.0)
