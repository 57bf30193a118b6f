"""The N > 1 path of bench.py on CPU: world size 2 over gloo (127.0.0.1).

The layer has no data-path collective (replicas only); what runs across ranks
is the bench's barrier, the max over ranks of the timed span and the sum over
ranks of the work, and the reference arm's rank-0-only line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, out_dir: str):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    world, r, local = bench.dist_setup()
    bench.barrier(world)
    mx = bench.reduce_max(1.5 + 2.0 * r, world)      # rank 0: 1.5, rank 1: 3.5
    sm = bench.reduce_sum(10.0 * (r + 1), world)     # 10 + 20
    bench.barrier(world)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": world, "rank": r, "local": local, "max": mx, "sum": sm}, f)
    import torch.distributed as dist

    dist.destroy_process_group()


def test_reductions_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        d = json.load(open(tmp_path / f"rank{r}.json"))
        assert d == {"world": 2, "rank": r, "local": r, "max": 3.5, "sum": 30.0}


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--gpus", "2", "--tokens", "1", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
