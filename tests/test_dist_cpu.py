"""The multi-process path of bench.py on CPU (gloo, world size 2): the host
timing exchange (max over ranks, barrier) and the replica launch under
torchrun, where rank 0 alone prints the JSON line.  The library path has no
collective: N GPUs run N independent replicas."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.dist_barrier(w)
    got = bench.dist_max(1.5 + rank, w)
    dist.destroy_process_group()
    with open(os.path.join(out, "rank%d" % rank), "w") as f:
        f.write(repr(got))


def test_timing_max_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    mp.spawn(_worker, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        assert float((tmp_path / ("rank%d" % rank)).read_text()) == 2.5


def test_reference_arm_under_torchrun_prints_one_line():
    """torchrun with two ranks: rank 0 times the oracle sample and prints the
    reference line; rank 1 does no work and exits 0."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--ref-rows", "1"]
    p = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    for key in ("metric", "unit", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data"):
        assert key in d, key
    # the same workload, metric and unit as the GPU arm's line
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"] == bench.workload_config(2)
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"]
