"""The multi-GPU path of bench.py is replicas only: every rank runs its own blend and the job's
throughput is (ranks x units) / slowest rank.  Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    ws_, rank_, local_ = bench.dist_setup(None)
    assert (ws_, rank_, local_) == (ws, rank, rank)
    bench.barrier(ws)
    local_ms = [1000.0, 1500.0][rank]          # rank 1 is the slower replica
    value, ms_per_step = bench.replica_throughput(ws, 3072, 10, local_ms)
    out[rank] = (value, ms_per_step)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replica_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # both ranks agree: 2 replicas x 3072 tokens x 10 steps over the slower rank's 1.5 s
    for r in range(2):
        value, ms = out[r]
        assert abs(value - 2 * 3072 * 10 / 1.5) < 1e-6
        assert abs(ms - 150.0) < 1e-9


def test_single_rank_needs_no_process_group():
    import bench
    value, ms = bench.replica_throughput(1, 100, 4, 200.0)
    assert value == pytest.approx(100 * 4 / 0.2) and ms == pytest.approx(50.0)


def test_blend_floor_takes_the_larger_bound_per_class():
    """Roofline time of a blend: per kernel class the larger of FLOPs / tensor peak and bytes / HBM peak."""
    import bench
    prof = [
        {"name": "gemm", "flops": 2 * 1e12, "bytes": 2 * 1e9},     # per step: 1 TFLOP -> 1 ms at 1000 TF/s
        {"name": "copy", "flops": 0, "bytes": 2 * 5e9},             # per step: 5 GB -> 1 ms at 5000 GB/s
        {"name": "mixed", "flops": 2 * 1e9, "bytes": 2 * 10e9},     # bytes bound: 2 ms
    ]
    assert abs(bench.blend_floor_ms(prof, 2, 1000.0, 5000.0) - 4.0) < 1e-9
    # no tensor peak (fp32 configuration): bytes only
    assert abs(bench.blend_floor_ms(prof, 2, None, 5000.0) - (0.2 + 1.0 + 2.0)) < 1e-9


def test_traffic_lookup_needs_matching_workload_and_source():
    """The committed DRAM-traffic figure of a kernel is used only for the workload it was captured on,
    and only while the kernel's source is the one it was taken from."""
    import json
    import os
    import bench
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")))
    for key, ent in d.items():
        kernel = key.split("@")[0]                  # "kernel" or "kernel@workload"
        got = bench.load_traffic(kernel, ent["workload"])
        assert got in (None, ent["dram_bytes_per_launch_full"])
        captured = {e["workload"] for k, e in d.items() if k.split("@")[0] == kernel}
        for other in ("llama8b-3k", "llama8b-8k", "llama8b-32k"):
            if other not in captured:
                assert bench.load_traffic(kernel, other) is None
    assert bench.load_traffic("no-such-kernel", "llama8b-3k") is None
