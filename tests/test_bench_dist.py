"""The bench's multi-rank host logic on CPU: two gloo ranks (127.0.0.1) check
the max/sum-over-ranks aggregation used for the timed region and that only
rank 0 runs and prints the reference arm."""
import io
import os
import socket
import contextlib

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(10.0 * (rank + 1))
        sm = bench.sum_over_ranks(rank + 1)
        bench.dist_barrier()
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                            "--ref-step-seconds", "0.05"])
        q.put((rank, mx, sm, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_rank_aggregation_gloo_world_size_2():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(world))
    for rank, mx, sm, out in results:
        assert mx == 20.0
        assert sm == 3.0
        if rank != 0:
            assert out == ""      # the reference arm runs on rank 0 only


def test_single_process_aggregation_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.sum_over_ranks(2) == 2.0


def test_reference_arm_prints_one_json_line(capsys):
    import json
    import bench
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                "--ref-step-seconds", "0.05"])
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
