"""The benchmark's multi-process path (one replica per rank, slowest rank's
time, whole-job throughput) on CPU with gloo, world size 2."""
import json
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, w)   # rank 1 is slower
    value = bench.job_throughput(1000, w, slowest)
    # the reference arm runs on rank 0 only; other ranks return without work
    ref = bench.run_reference(type("A", (), {"workload": bench.DEFAULT_WORKLOAD, "steps": 1,
                                             "warmup": 0, "cpu_seconds": 1.0})(), w, r) \
        if r != 0 else "skipped"
    with open(os.path.join(out_dir, "rank%d.json" % r), "w") as f:
        json.dump({"world": w, "slowest": slowest, "value": value, "ref": ref}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_gloo(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    for x in res:
        assert x["world"] == 2
        assert x["slowest"] == 15.0          # max over ranks
        assert abs(x["value"] - 1000 * 2 / 15e-3) < 1e-6
    assert res[1]["ref"] is None             # non-zero ranks print nothing
