"""The multi-rank host logic of bench.py on 2 gloo ranks (CPU, no GPU): every
rank draws its own batch, the slowest rank sets the time, and the whole-job
value counts every rank's bytes.  The reference arm prints on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from kimi_k3_attention_gb300 import workloads as wl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # distinct batches per rank
        inp = wl.make_inputs(2, 1, 16, seed=bench.rank_seed(rank))
        t_rank = 0.010 * (rank + 1)          # rank 1 is the slow one
        t = bench.max_over_ranks(t_rank, "cpu")
        v = bench.weak_scaling_value(1000, world, 5, t)
        q.put((rank, t, v, inp.prefix.float().sum().item()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, v0, s0), (r1, t1, v1, s1) = res
    assert t0 == t1 == pytest.approx(0.020)
    assert v0 == v1 == pytest.approx(1000 * 2 * 5 / 0.020 / 1e9)
    assert s0 != s1


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_gpus_flag_starts_the_ranks_itself():
    """`bench.py --gpus 2` outside a launcher starts two ranks on this node
    (torch.distributed.run); the dry run exercises the rank set-up, barriers,
    timing and max over ranks with gloo and no GPU: exactly one line, from
    rank 0, with n_gpus 2 and the slower rank's time."""
    import json
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--dry-run", "--gpus", "2",
                        "--steps", "5", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["dry_run"] and d["scaling"] == "weak"
    assert d["ms_per_step"] >= 2.0          # rank 1 sleeps 2 ms per step


def test_gpus_flag_must_match_the_launcher():
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--dry-run", "--gpus", "4",
                        "--steps", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "WORLD_SIZE" in r.stderr
