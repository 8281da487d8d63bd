"""The N > 1 path of bench.py on CPU: world size 2 over gloo.

Each rank runs its own copy of the workload (the cases shard without
exchange), so the only cross-rank step is the timing: the job's time is the
slowest rank's, and the value counts every rank's bytes.  The reference arm
runs on rank 0 alone and prints one line.
"""

import json
import os
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    t = bench.max_over_ranks(10.0 + 5.0 * rank)     # rank 1 is slower
    v = bench.job_value(1_000_000_000, 2, world, t)
    out.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29613
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    # 2 ranks x 1 GB x 2 steps over 15 ms
    assert abs(res[0][2] - 2 * 1e9 * 2 / 0.015 / 1e9) < 1e-9


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", "29617", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "GB/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
