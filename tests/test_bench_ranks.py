"""bench.py's multi-process path on the CPU: replicas joined by a gloo process
group (world size 2), as the GPU bench runs them under torchrun with one
process per GPU.

* the rank set-up, barrier and max-over-ranks helpers the timed region uses;
* the whole-job aggregate (replicas x calls in the slowest rank's time);
* the reference arm under a 2-process torchrun: rank 0 alone prints one line.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w = bench.dist_setup("gloo")
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 * (rank + 1), w, "cpu")
    q.put((r, w, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 20.0), (1, 2, 20.0)]


def test_job_aggregate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas x 32 layer calls in the slowest rank's 1.6 ms -> 25 us per layer for the job
    assert abs(bench.job_us_per_layer(1.6, 32, 2) - 25.0) < 1e-12
    assert bench.job_us_per_layer(1.6, 32, 1) == 2 * bench.job_us_per_layer(1.6, 32, 2)


def test_reference_arm_under_two_ranks_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0", "--gpus", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
