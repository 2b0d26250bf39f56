"""The benchmark's multi-rank logic (replicas, max over ranks, whole-job
throughput) on CPU with two gloo ranks."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
    slow = bench.max_over_ranks(ms, world, "cpu")
    q.put((rank, slow, bench.aggregate_value(slow, 8192, world)))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, val in out:
        assert slow == 15.0
        assert abs(val - 2 * 8192 / 0.015) < 1e-6


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_value(2.0, 1000, 1) == 500000.0
    from grouped_gemm_moe_gb300 import workloads as W
    cfg = W.CONFIGS["qwen3"]
    fl, nb = bench.kernel_work("gemm_gate_up", cfg, False)
    assert fl == 4 * cfg.T * cfg.K * cfg.d * cfg.I
    # weights read once: 2 * E * d * I bf16 values are part of the bytes
    assert nb > 2 * cfg.E * cfg.d * cfg.I * 2
    pk = {"hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0, "bf16_tflops": 1900.0}
    assert bench.roofline_of(fl, 1.0, 1.0, pk)["bound"] == "tensor"
    assert bench.roofline_of(1.0, nb, 1.0, pk)["bound"] == "hbm"
