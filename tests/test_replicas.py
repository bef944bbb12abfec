"""The multi-rank host path of bench.py on CPU (gloo, world size 2): replicas
only, so the ranks exchange nothing but the timing reductions (a barrier, the
slowest rank's time, the sum of every rank's tokens), and the reference arm
prints one line from rank 0 while the other ranks exit without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")
# bench.py picks NCCL when a device is visible; these are the CPU (gloo) checks
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo replica checks run on CPU")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    w, r, _, pg = bench.dist_setup(None)
    try:
        bench.barrier(pg)
        t_max = bench.max_over_ranks(pg, 10.0 + rank)      # the slowest rank's time
        tokens = bench.sum_over_ranks(pg, 100.0 * (rank + 1))  # every rank's tokens
        bench.barrier(pg)
        out.put((r, w, t_max, tokens))
    finally:
        pg.destroy_process_group()


def test_rank_reductions_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    for _, w, t_max, tokens in got:
        assert w == world
        assert t_max == 11.0        # max over ranks
        assert tokens == 300.0      # sum over ranks


def test_reference_arm_prints_one_line_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
