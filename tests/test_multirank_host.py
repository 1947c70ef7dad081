"""The multi-rank host logic of bench.py on CPU with gloo, world size 2.

Each rank runs its own independent batch (weak scaling): the workloads differ by
seed, the timing reduction takes the maximum over ranks, the token count is the
sum over ranks, and the reference arm prints only on rank 0.  No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import bench
    import workloads
    w_env, r_env, _ = bench.dist_env()
    bench.init_dist(w_env)
    dev = torch.device("cpu")
    t_max = bench.max_over_ranks(10.0 + rank, w_env, dev)
    tok = bench.sum_over_ranks(float(100 * (rank + 1)), w_env, dev)
    bench.barrier(w_env)
    w = workloads.make("tiny", seed=r_env)
    q.put((rank, t_max, tok, int(w.q.view(-1)[0].view(torch.int16))))
    torch.distributed.destroy_process_group()


def test_two_rank_reductions_and_independent_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [11.0, 11.0]          # max over ranks
    assert [g[2] for g in got] == [300.0, 300.0]        # sum over ranks
    assert got[0][3] != got[1][3]                       # different seeds -> different data


def test_reference_arm_prints_once_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--config", "tiny"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
