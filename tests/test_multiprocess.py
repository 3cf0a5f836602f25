"""The N > 1 path of bench.py on CPU: world_size-2 gloo process groups.

The attention path shards by (request, kv head) with no exchange, so N GPUs
run N independent replicas; the only cross-rank steps are the barriers
around the timed region and the max-over-ranks of the step time.  These
tests run them as two gloo ranks (127.0.0.1), and run the bench's
reference arm under torchrun, where rank 0 alone prints the JSON line.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench._dist()
    bench._barrier(w)
    m = bench._max_over_ranks(1.5 + r, w)
    bench._barrier(w)
    queue.put((r, w, local, m, dist.get_backend()))
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[:3] for r in results] == [(0, 2, 0), (1, 2, 1)]
    assert all(r[3] == 2.5 for r in results)          # the slower rank's time wins
    assert all(r[4] == "gloo" for r in results)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "1", "--steps", "1",
           "--warmup", "3"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_line_keeps_the_contract():
    """One rank: the reference arm's JSON line carries the keys the driver
    reads, with the oracle as its CPU baseline and zero host transfers."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "1", "--steps", "2",
           "--warmup", "3"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "impl"):
        assert k in res, k
    assert res["n_gpus"] == 1 and res["steps"] == 2 and res["warmup"] == 3
    assert res["e2e"]["value"] == res["value"]
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["d2h_bytes_per_step"] == 0
    assert res["cpu_baseline"]["value"] == res["value"] and res["cpu_baseline"]["cores"] >= 1
