"""Several ranks, one process each (replicas: the encode has no data-path
collective, each rank encodes its own batch): the host side of bench.py's
N > 1 path, on CPU with the gloo backend."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each rank's step time differs; the job's time is the slowest rank's
    v = bench.max_over_ranks(1.5 + rank, world, device="cpu")
    single = bench.max_over_ranks(7.0, 1, device="cpu")
    dist.barrier()
    with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
        f.write(f"{v!r} {single!r}")
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    got = [open(tmp_path / f"r{r}").read().split() for r in range(2)]
    assert got == [["2.5", "7.0"], ["2.5", "7.0"]]


def test_replica_batches_differ_per_rank():
    """Weak scaling: every rank encodes a batch of the same size and shape
    from its own seed."""
    sys.path.insert(0, ROOT)
    import bench
    a = bench.make_workload("prose", 0)
    b = bench.make_workload("prose", 1)
    assert a[1].size == b[1].size and a[2].size == b[2].size
    assert not np.array_equal(a[1], b[1])


def test_reference_arm_under_torchrun():
    """`bench.py --impl reference` launched like the driver launches N > 1:
    rank 0 alone times the oracle and prints the one JSON line; rank 1 exits
    0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "prose"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the sample is stated, and the oracle ran pinned to one core
    assert d["cpu_baseline"]["pinned_cores"] is not None and len(d["cpu_baseline"]["pinned_cores"]) == 1
    assert "segments 0..0" in d["cpu_baseline"]["sample"] and d["cpu_baseline"]["host_cpu"]["nproc"] >= 1
