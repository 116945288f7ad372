"""Host-side logic of bench.py, without a GPU: the reference (oracle) arm's
JSON line, its rank handling under torchrun, and the max-over-ranks timing
reduction across two gloo ranks."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_json_line():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "diag-bf16-b8h16t4096d128"


def test_reference_arm_other_ranks_exit_without_work():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "0", "--gpus", "2"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mx = bench.reduce_max(torch, dist, 10.0 + 5 * rank, world, torch.device("cpu"))
    q.put((rank, mx, bench.aggregate_tokens_per_s(1000, mx, world)))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]              # slowest rank's ms on every rank
    assert res[0][2] == pytest.approx(2 * 1000 / 0.015)      # all ranks' tokens / slowest time


def test_reference_arm_pkda_workload():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "pkda-bf16-b8h16t4096d128"])
    assert r.returncode == 0, r.stderr
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["config"]["workload"] == "pkda-bf16-b8h16t4096d128"
