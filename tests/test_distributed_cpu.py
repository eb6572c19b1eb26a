"""The multi-GPU path of bench.py on the CPU (no GPU).

The layer does not shard across GPUs (replicas only): with N ranks every rank runs the
same steps on its own GPU, the timed region is the slowest rank's, and the job's value
is the tokens of all ranks over that time. Here two gloo ranks (127.0.0.1) check the
max-over-ranks reduction and the whole-job value, and the reference arm under torchrun
with two processes checks that rank 0 alone runs and prints and rank 1 exits 0.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, ws)
    value = bench.job_tokens_per_s(64 * 50, ws, ms)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in got:
        assert ms == 15.0                              # both ranks see the slowest time
        assert value == pytest.approx(64 * 50 * 2 / 0.015)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--ref-tokens", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2
    assert out["cpu_baseline"]["kind"] == "oracle" and out["value"] > 0
    assert out["e2e"]["h2d_bytes_per_step"] == 0
