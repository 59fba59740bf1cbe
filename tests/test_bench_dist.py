"""bench.py's multi-rank logic on the CPU, world size 2 over gloo: the
slowest rank's time, the sum of all ranks' units, and the reference arm
printing one JSON line from rank 0 only."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import bench
    ms, value = bench.aggregate(1.0 + 2.0 * rank, 100.0 + rank, world=2)
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_aggregate_takes_slowest_rank_and_sums_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 3.0                         # max(1.0, 3.0)
        assert abs(value - 201.0 / 3e-3) < 1e-6  # (100 + 101) units / 3 ms


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--ref-sample", "8192"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_oracle_split_over_threads_gives_the_same_bits():
    """The CPU baseline's threaded form (contiguous chunks, one oracle call
    each) leaves master/m/v bit-identical to one call over the sample."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    runs = []
    for threads in (1, 3, 8):
        g16, st, hp, n = bench.oracle_sample_inputs(4, 10_007)
        runner = bench.OracleRunner(g16, st, hp, threads)
        assert len(runner.chunks) == threads
        assert sum(c[1][0].size for c in runner.chunks) == n
        runner.step()
        runner.step()
        runner.close()
        runs.append([x.view(np.uint32).copy() for x in st])
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert np.array_equal(a, b)
