"""The benchmark's multi-process path on CPU (gloo, world size 2): process-group
setup, the barrier around the timed region, the maximum of the step time over
ranks, and the reference arm's rule that only rank 0 runs and prints.
Decode sequences shard across ranks with no data-path collective, so these
host-side steps are the whole of the multi-GPU path."""
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_WORKER = r"""
import json, sys
sys.path.insert(0, {root!r})
import bench
rank, world = bench._dist_init()
bench._barrier(world)
m = bench._max_over_ranks(1.5 + rank, world)
bench._barrier(world)
import torch.distributed as dist
print(json.dumps({{"rank": rank, "world": world, "max": m, "backend": dist.get_backend()}}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _env(rank, world, port):
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    return env


def test_two_ranks_barrier_and_max_over_ranks():
    import json
    port = _free_port()
    code = _WORKER.format(root=ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code], cwd=ROOT, env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["world"] == 2 and o["backend"] == "gloo"
        assert o["max"] == 2.5  # max over ranks of 1.5 + rank


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun every rank but 0 leaves the reference arm at once,
    without output and without joining a process group."""
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=_env(1, 2, _free_port()), capture_output=True, text=True, timeout=180)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
