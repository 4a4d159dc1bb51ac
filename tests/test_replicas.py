"""Multi-GPU path = independent replicas over disjoint requests (the units of
the path share nothing), timed as the slowest rank.  Checked here with two
gloo ranks on the CPU."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from synth import workloads as W
    w = W.make("attention", R=4, steps=3)
    w.req_base = bench.replica_request_base(rank, w.R)
    tr = np.stack([w.trace(r) for r in range(w.R)])
    slow = bench.max_over_ranks(10.0 + 5.0 * rank, dist)       # rank 1 is slower
    rate = bench.weak_scaling_rate(w.L * w.R * w.K, 7, world, slow)
    out[rank] = (w.req_base, tr.sum(), slow, rate)
    dist.destroy_process_group()


def test_two_gloo_replicas_partition_requests_and_time_the_slowest():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    (b0, s0, t0, r0), (b1, s1, t1, r1) = out[0], out[1]
    assert (b0, b1) == (0, 4)                  # disjoint requests per replica
    assert s0 != s1                            # hence different selection traces
    assert t0 == t1 == 15.0                    # both report the slowest rank
    assert r0 == r1 == world * 7 * (2 * 4 * 2048) / 15e-3


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_request_base(3, 32) == 96


def test_bench_spawns_one_replica_per_gpu_with_disjoint_requests():
    """`bench.py --gpus 2` outside torchrun relaunches itself as two ranks
    (gloo here, no GPU work: --replica-check); rank 0 reports both replicas'
    request ranges, which are disjoint, and n_gpus = 2."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--replica-check"], capture_output=True, text=True, timeout=300,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    (a0, a1), (b0, b1) = line["replica_requests"]
    per = line["requests_per_replica"]
    assert (a0, a1, b0, b1) == (0, per, per, 2 * per)
