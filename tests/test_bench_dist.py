"""bench.py's multi-rank path on the CPU: two gloo ranks (no GPU needed).

The per-GPU path shards by replicas (every rank runs the same workload, no collective
on the data path); what crosses ranks is the timing: a barrier on both sides of the
timed region, the max over ranks of the elapsed time, and the whole-job throughput
computed from it.  These tests run that plumbing with world_size 2 over gloo, and the
reference arm under torchrun, where rank 0 alone prints the JSON line.
"""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # per-rank elapsed times 1.5 s and 2.5 s: the job takes as long as its slowest rank
    t_max = bench.max_over_ranks(1.5 + rank, w)
    value = bench.aggregate_value(1000.0, w, t_max)
    bench.barrier(w)
    Path(out_dir, f"rank{rank}.json").write_text(json.dumps({"t_max": t_max, "value": value}))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_max_and_aggregate(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(world)]
    for r in res:
        assert r["t_max"] == 2.5
        # 1000 units per rank, 2 ranks, 2.5 s: whole-job throughput 800 units/s
        assert r["value"] == pytest.approx(800.0)


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(ROOT / "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "c1_small_f32"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
