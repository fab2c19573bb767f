"""The N > 1 path of bench.py on CPU: two gloo ranks rendezvous on 127.0.0.1, time
independent replicas and agree on the slowest rank's time (max over ranks), with no
collective on the data path."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, time
sys.path.insert(0, {root!r})
import bench
rank, world, local = bench.dist_setup(2)
assert world == 2 and rank == int(os.environ["RANK"])
bench.barrier(world)
# each rank "times" its own replica; the reported time is the slowest rank's
t = 1.0 + rank
tmax = bench.max_over_ranks(t, world)
assert tmax == 2.0, tmax
bench.barrier(world)
print(f"rank {{rank}} ok {{tmax}}")
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_max_time(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = []
    for p in procs:
        try:
            out, _ = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("gloo rank hung")
        outs.append(out)
        assert p.returncode == 0, out
    assert "rank 0 ok 2.0" in outs[0] and "rank 1 ok 2.0" in outs[1]


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs the oracle reference arm; other ranks return."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
