"""bench.py's multi-process path (replicas): the max-over-ranks elapsed time
and the sum of units, with world_size 2 gloo ranks on the CPU."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    el, units = bench.reduce_over_ranks(1.0 + rank, 10.0 * (rank + 1))
    bench.barrier()
    q.put((rank, el, units))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_reduce_over_ranks_gloo(world):
    import socket

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, el, units in res:
        assert el == 2.0            # max over ranks
        assert units == 30.0        # 10 + 20


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_over_ranks(1.5, 7.0) == (1.5, 7.0)


def test_multi_gpu_refused_before_the_library_loads_for_multicast_workloads():
    """The CTA-pair GEMMs load with cluster-multicast TMA, which runs only in
    single-GPU calls: with WORLD_SIZE 2, bench.py prints an "unavailable" line
    for a workload that reaches them and exits 0 before importing the package
    (so libfp8blk.so is never loaded)."""
    import json
    import subprocess

    code = (
        "import runpy, sys\n"
        "sys.argv = ['bench.py', '--gpus', '2', '--workload', 'prefill_gemm_w1', '--steps', '3', '--warmup', '3']\n"
        "try:\n"
        "    runpy.run_path('bench.py', run_name='__main__')\n"
        "except SystemExit as e:\n"
        "    assert not e.code, e.code\n"
        "assert 'fp8_block_scaled_quant_gb300' not in sys.modules\n"
        "assert 'torch' not in sys.modules\n"
    )
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "ours" and "unavailable" in line


def test_replica_workloads_never_plan_cluster_pairs():
    """Every workload bench.py runs as multi-GPU replicas keeps its GEMMs on
    plans without cluster pairs (mirror of the library's plan)."""
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    from test_gemm_schedule import make_plan

    for name, (kind, shape) in bench.WORKLOADS.items():
        if bench.reaches_cluster_multicast(kind, shape) or kind != "linear":
            continue
        for sms in (148, 152, 160):
            assert make_plan(shape["M"], shape["N"], shape["K"], sms)["cluster"] == 1, name
