"""Host-side logic of the multi-GPU benchmark, on CPU with a world-size-2 gloo group.

Requests are independent, so every rank resolves its own requests (weak scaling) and
the only collective is the max of the ranks' timings; no collective touches the data.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import tracegen
    local = [10.0 + 5 * rank, 100.0 - rank]
    got = bench.reduce_max(local, dist, "cpu")
    w = bench.workload_for_rank("dsa", rank)
    sel = tracegen.trace(w, T=2, B=2)
    np.save(os.path.join(out_dir, f"sel{rank}.npy"), sel)
    with open(os.path.join(out_dir, f"max{rank}.txt"), "w") as f:
        f.write(" ".join(str(x) for x in got))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_shard_requests_and_take_the_max(tmp_path):
    import tracegen
    tracegen.build()
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        vals = [float(x) for x in open(tmp_path / f"max{r}.txt").read().split()]
        assert vals == [15.0, 100.0]
    s0, s1 = np.load(tmp_path / "sel0.npy"), np.load(tmp_path / "sel1.npy")
    assert not np.array_equal(s0, s1)          # each rank resolves different requests
    w = tracegen.WORKLOADS["dsa"]
    assert np.array_equal(s0, tracegen.trace(w, T=2, B=2))  # rank 0 is the configured workload


def test_weak_scaling_value_counts_every_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.weak_scaling_value(1, 32, 10, 1000.0) == pytest.approx(320.0)
    assert bench.weak_scaling_value(4, 32, 10, 1000.0) == pytest.approx(1280.0)
    assert bench.reduce_max([1, 2], None, "cpu") == [1.0, 2.0]


def test_kernel_code_digest_ignores_comments_only(tmp_path):
    """The profile figures are keyed to the kernel code: a comment or whitespace edit keeps
    the key, a code edit changes it."""
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// header\n__global__ void k(int* p) { /* note */ p[0] = 1; }\n")
    b = tmp_path / "b.cu"
    b.write_text("// another header\n\n__global__ void k(int* p) {\n    p[0] = 1;  // same code\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.kernel_code_digest(str(a)) == bench.kernel_code_digest(str(b))
    assert bench.kernel_code_digest(str(a)) != bench.kernel_code_digest(str(c))


def test_reference_arm_under_two_ranks_prints_one_line():
    """`bench.py --impl reference` launched as the driver launches it for N = 2: one JSON
    line from rank 0 with the reference arm's keys, the other rank exits 0 without output."""
    import json
    import subprocess
    import sys
    import oracle
    import tracegen
    oracle.build()
    tracegen.build()
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "tiny"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
