"""The bench's multi-process path on the CPU: two ranks over gloo (127.0.0.1).
Each GPU runs an independent replica of the whole simulated domain (its own
microbatch), so the only cross-rank steps are the barrier around the timed
region and the max over ranks of the elapsed time; the reference arm runs on
rank 0 alone.  No GPU is used."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    # CPU only, whatever machine runs the test: the ranks pick gloo
    os.environ.update(CUDA_VISIBLE_DEVICES="", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import types

    import torch
    import torch.distributed as dist

    import bench
    from moe_expert_load_id_b300 import workload as W

    r, w, local = bench.dist_init()
    res = {"rank": r, "world": w, "backend": dist.get_backend()}
    # each rank's elapsed time differs; all of them must report the slowest
    res["max"] = bench.max_over_ranks(10.0 * (r + 1), w, torch.device("cpu"))
    bench.barrier(w)
    # the reference arm (the CPU oracle) runs on rank 0 only
    args = types.SimpleNamespace(w=W.WORKLOADS["tiny"], workload="tiny", steps=1, warmup=3)
    line = bench.run_reference(args, r, w)
    res["reference"] = None if line is None else (line["impl"], line["n_gpus"],
                                                   line["cpu_baseline"]["kind"])
    bench.barrier(w)
    dist.destroy_process_group()
    out.put(res)


def test_two_ranks_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda d: d["rank"])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [d["world"] for d in res] == [2, 2]
    assert all(d["backend"] == "gloo" for d in res)
    assert [d["max"] for d in res] == [20.0, 20.0]
    assert res[0]["reference"] == ("reference", 2, "oracle")
    assert res[1]["reference"] is None


def test_whole_job_metric():
    sys.path.insert(0, ROOT)
    import bench
    # two replicas, 5 steps of 94 layers each, slowest rank 1640 ms in all
    assert bench.whole_job_us_per_layer(1640.0, 5, 94, 2) == pytest.approx(1640e3 / (5 * 94 * 2))
    assert bench.whole_job_us_per_layer(10.0, 1, 1, 1) == pytest.approx(10000.0)
