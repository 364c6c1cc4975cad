"""Host-side logic of the multi-rank benchmark, on CPU with the gloo backend (world size 2):
the slowest rank's time is used and the job value counts every rank's units."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        bench.barrier()
        my_ms = 100.0 + 50.0 * rank  # rank 1 is slower
        mx = bench.max_over_ranks(my_ms)
        val = bench.job_throughput(2.0e9, ws, 10, mx)
        q.put((r, local, ws, mx, val))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, local, ws, mx, val) in enumerate(res):
        assert rank == r and local == r and ws == 2
        assert mx == 150.0
        assert val == pytest.approx(2.0e9 * 2 * 10 / 0.150)


def test_single_process_helpers():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(1e12, 1, 4, 1000.0) == pytest.approx(4e12)
    from mixture_experts_forward_moe_gb300 import inputs
    w = inputs.WORKLOADS["qwen3-30b-a3b-decode-t32"]
    ab = bench.algorithmic_bytes(w, 112)
    assert ab["total"] == 112 * 3 * 768 * 2048 * 2 + 32 * 2048 * 2 * 2 + 32 * 128 * 4


def test_kernel_hash_ignores_comments_but_not_code():
    src = "int a = 1;  // one\n/* a block\n   comment */\n\nint b = 2;\n"
    assert bench._code_only(src) == "int a = 1;\nint b = 2;"
    assert bench._code_only(src.replace("// one", "// uno")) == bench._code_only(src)
    assert bench._code_only(src.replace("b = 2", "b = 3")) != bench._code_only(src)


def test_recorded_traffic_only_for_the_captured_kernels(monkeypatch):
    import json
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    wl, per = next(iter(rec["per_launch_bytes"].items()))
    stage, nbytes = next(iter(per.items()))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["kernel_source_hash"])
    assert bench.recorded_traffic(wl, stage) == nbytes
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic(wl, stage) is None
