"""The benchmark's multi-process (one rank per GPU) host logic, on the CPU with two gloo ranks:
max-over-ranks timing, the whole-job value, and the reference arm running on rank 0 alone."""
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tiny_workloads(seed=0):
    import bench
    import synth
    w = synth.make_dense(4, 256, 256, seed=seed)
    w["name"] = "dense_4x256x256"
    w["valid_rows"] = bench._valid_rows(w)
    w["flops"] = 2.0 * w["valid_rows"] * w["N"] * w["K"]
    w["bytes"] = bench._algorithmic_bytes(w)
    return [w]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
        value = bench.whole_job_tflops(1e12, 10, world, slowest)
        bench.make_workloads = _tiny_workloads
        out = bench.run_reference(types.SimpleNamespace(steps=1, warmup=0), rank, world)
        dist.barrier()
        q.put((rank, slowest, value, out))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, slowest, value, out = q.get(timeout=120)
        res[rank] = (slowest, value, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time; the value counts both replicas' work
    assert res[0][0] == res[1][0] == 20.0
    assert res[0][1] == pytest.approx(2 * 1e12 * 10 / 20e-3 / 1e12)
    # the reference arm works on rank 0 only
    assert res[1][2] is None
    out = res[0][2]
    assert out["impl"] == "reference" and out["n_gpus"] == world and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle"
