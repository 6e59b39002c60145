"""bench.py with several ranks, on CPU (gloo, world_size 2): the barrier and the max over ranks
that the timed regions use, and the reference arm under torchrun (rank 0 prints the one JSON line,
the other ranks exit 0 without work).  The layer itself runs as independent replicas (no
data-path collective), so these are the only multi-rank code paths."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    torch.cuda.is_available = lambda: False  # gloo even where a GPU is visible
    import bench
    r, w, _ = bench._dist()
    bench._barrier(w)
    m = bench._max_over_ranks(float(rank) + 0.5, w)
    bench._barrier(w)
    q.put((r, w, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(60)
    assert res == [(0, 2, 1.5), (1, 2, 1.5)]
    assert all(p.exitcode == 0 for p in procs)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2",
           "--warmup", "3", "--workload", "tiny"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
