"""The multi-process paths of bench.py on CPU (gloo, world size 2): the
max-over-ranks timing helper and barrier, and the reference arm launched the
way the driver launches N > 1 (torch.distributed.run, rank 0 alone prints)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    bench.barrier(dist)
    got = bench.allreduce_max(dist, 1.5 + rank)
    bench.barrier(dist)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo(tmp_path):
    import torch
    import torch.multiprocessing as mp
    if torch.cuda.is_available():
        pytest.skip("the helper reduces on the GPU when one is present")
    mp.start_processes(_worker, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 2.5


def test_reference_arm_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--cpu-seconds", "0.2", "--workload", "na3d_b1_t4_h8_w16_nh2_hd32_k3x5x5"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
