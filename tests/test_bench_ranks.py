"""The multi-rank host logic of bench.py on CPU: two gloo ranks meet at the
barrier, take the slowest rank's time (all-reduce MAX) and report the
whole-job rate; under the reference arm only rank 0 works.  No GPU: the same
functions run over NCCL on GPUs, with the scalar on the device."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, ws, port, out):
    import torch.distributed as tdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    tdist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        ms = [3.5, 2.0][rank]                       # rank 0 is the slower one
        slowest = bench.max_over_ranks(ms, ws, "cpu")
        out.put((rank, slowest, bench.whole_job_rate(64, ws, slowest)))
        bench.barrier(ws)
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]
    assert all(r[2] == pytest.approx(2 * 64 / 3.5e-3) for r in res)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.whole_job_rate(8192, 1, 2.0) == pytest.approx(8192 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload, steps, warmup = "tiny", 1, 0
    bench.run_reference(A(), 2, 1)                  # rank 1 of 2: no work, no output
    assert capsys.readouterr().out == ""


def test_bench_gpus_2_starts_two_ranks():
    """`python bench.py --gpus 2` started as one process re-launches itself
    as two local ranks (torch.distributed.run); here in the launcher
    self-test mode, where the ranks meet over gloo without a GPU and rank 0
    alone prints one line reporting both ranks."""
    import json
    import subprocess
    env = dict(os.environ)
    for v in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(v, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--launch-selftest"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and rec["ranks_seen"] == 2 and rec["slowest_rank_value"] == 2.0
