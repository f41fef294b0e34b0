"""The N > 1 path of bench.py on the CPU: one process per rank over gloo,
world size 2.  The workload does not shard (every rank runs an independent
replica), so the only cross-rank steps are the barrier around the timed
region and the max over ranks of the elapsed time; both are checked here,
together with the whole-job aggregation (all ranks' units / the max time)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(world)
    d.barrier()
    # rank r "took" 10 + r ms for one unit of work
    ms = d.max(10.0 + rank)
    value = bench.job_value(units_per_rank=1.0, world=d.world, ms=ms)
    d.barrier()
    d.close()
    out.put((rank, d.world, ms, value))


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    for _, world, ms, value in res:
        assert world == 2
        assert ms == 11.0                       # the slowest rank's time, on every rank
        assert value == pytest.approx(2.0 / 11e-3)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    old = {k: os.environ.pop(k, None) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    try:
        d = bench.Dist(1)
        assert d.world == 1 and d.pg is None
        assert d.max(3.5) == 3.5
        d.barrier()
        d.close()
        assert bench.job_value(units_per_rank=4.0, world=1, ms=2.0) == pytest.approx(2000.0)
    finally:
        for k, v in old.items():
            if v is not None:
                os.environ[k] = v


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched as the benchmark driver launches
    it for N = 2: rank 0 alone times the oracle and prints one JSON line;
    rank 1 exits 0 without output."""
    import json
    import subprocess
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
