"""bench.py's multi-GPU path (a real ring over the job's ranks) run end to
end: two ranks under torchrun sharing this GPU, the K/V blocks exchanged over
gloo through pinned host memory (CP_BENCH_BACKEND=gloo).  With NCCL and one
GPU per rank the same code moves the blocks GPU to GPU; this checks the
driver loop, the three timings, the end-to-end leg and the JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_bench_ring_two_ranks_over_gloo(cuda_dev):
    env = dict(os.environ, CP_BENCH_BACKEND="gloo")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--gpus",
           "2", "--steps", "2", "--warmup", "3", "--workload", "s8192"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["n_gpus"] == 2 and line["scaling"] == "strong"
    assert line["config"]["N_virtual_ranks"] == 2
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["e2e"]["value"] > 0
    ring = line["ring"]
    assert ring["ms_ring"] > 0 and ring["ms_compute"] > 0 and ring["ms_transfers"] > 0
    assert ring["hop_bytes"] == 2 * 1 * 4096 * 8 * 128 * 2      # k and v shards of one rank
    assert line["gpu_launches"] == 2 * 2
