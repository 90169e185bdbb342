"""The benchmark's multi-process path on CPU (gloo, world size 2): every rank
runs its own replica (the decode path has no exchange step), the timing is the
maximum over ranks and counts are summed; rank 0 alone prints."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dev = torch.device("cpu")
        bench.barrier(world)
        mx = bench.max_over_ranks(10.0 + rank, world, dev)
        sm = bench.sum_over_ranks(1.0, world, dev)
        q.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_sum_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0, 2.0), (1, 11.0, 2.0)]


def test_single_process_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.sum_over_ranks(2.0, 1, torch.device("cpu")) == 2.0
    bench.barrier(1)


def test_reference_arm_runs_on_rank0_only():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, workload, band_r, ref_budget = 2, 3, "gqa_4k_b1_contig", 64, 5.0
    assert bench.bench_reference(A(), 2, 1, 1) is None


def test_launch_count_and_traffic_provenance(tmp_path):
    """bench.py's claims about itself: a decode step is three launches, four
    with the grid-wide ring scan (rings over 32 entries) and one more with the
    side-stream Amend; the ncu traffic figure is used only while the hash of
    the attention kernel's sources matches the one the summary records."""
    sys.path.insert(0, ROOT)
    import bench
    from types import SimpleNamespace as NS
    assert bench.launches_per_step(NS(ring_len=16, group=32), 0) == 3
    assert bench.launches_per_step(NS(ring_len=32, group=4), 0) == 3
    assert bench.launches_per_step(NS(ring_len=33, group=4), 0) == 4
    assert bench.launches_per_step(NS(ring_len=1024, group=32), 1) == 5
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    h1 = bench.kernel_source_sha([str(src)])
    src.write_text("kernel v2")
    assert bench.kernel_source_sha([str(src)]) != h1 and len(h1) == 16
    assert any(f.endswith("mac_attention.cu") for f in bench.KERNEL_SOURCES)
    rec = tmp_path / "cap.json"
    rec.write_text(json.dumps({"kernel_source_sha256_16": h1, "traffic_bytes_per_launch": 123.0}))
    assert bench.profiled_traffic([str(src)], str(rec)) is None      # sources changed since the capture
    src.write_text("kernel v1")
    assert bench.profiled_traffic([str(src)], str(rec)) == 123.0
    assert bench.profiled_traffic([str(src)], str(tmp_path / "absent.json")) is None
