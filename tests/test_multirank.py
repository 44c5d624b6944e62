"""The benchmark's multi-rank plumbing on CPU (gloo, two ranks).

Each rank is an independent replica (the operator has no exchange step on
one GPU per process); the only cross-rank work is combining the timings:
the whole-job figure is the units of all ranks over the slowest rank's time.
The reference arm runs on rank 0 alone.
"""

import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _combine_worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    secs = [0.5, 0.8][rank]
    nbytes = [1.0e9, 2.0e9][rank]
    lookups = [10e6, 30e6][rank]
    q.put((rank, bench.combine_ranks(secs, nbytes, lookups, steps=4, device="cpu")))
    dist.barrier()
    dist.destroy_process_group()


def test_combine_ranks_two_gloo_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_combine_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):  # every rank sees the same whole-job numbers
        assert got[r]["value"] == pytest.approx(3.0e9 / 0.8 / 1e9)
        assert got[r]["lookups_per_s_M"] == pytest.approx(40e6 / 0.8 / 1e6)
        assert got[r]["ms_per_step"] == pytest.approx(1e3 * 0.8 / 4)


def _bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env, cwd=ROOT,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _bench({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}, "--impl", "reference", "--gpus", "2")
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _bench({"RANK": "0", "LOCAL_RANK": "0", "WORLD_SIZE": "2"}, "--impl", "reference", "--gpus", "2",
                "--workload", "tiny", "--steps", "2", "--warmup", "1")
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_cpu_baseline_reports_all_cores_and_one_thread():
    sys.path.insert(0, ROOT)
    import bench

    d = bench.cpu_baseline("tiny", seconds=0.05, single_steps=1)
    assert d["kind"] == "oracle" and d["value"] > 0 and d["cores"] >= 1
    assert d["single_thread"]["cores"] == 1 and d["single_thread"]["value"] > 0
