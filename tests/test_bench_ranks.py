"""The replica path of bench.py on CPU ranks (gloo, world size 2): the timed
region is the slowest rank's, throughput counts every rank's bytes, and only
rank 0 runs the reference arm."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 40.0][rank]
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        gbs = bench.job_gbs(1.0e9, 4, world, ms)
        ref = bench.run_reference(type("A", (), {"reference_rows": 2, "warmup": 3, "steps": 1})(),
                                  rank, world) if rank == 1 else None
        out.put((rank, ms, gbs, ref))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world_2():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs, ref in results:
        assert ms == 40.0, "every rank sees the slowest rank's time"
        assert gbs == pytest.approx(2 * 1.0e9 * 4 / 0.040 / 1e9)
    assert results[1][3] is None, "a rank other than 0 does no reference work"


def test_single_rank_is_the_identity():
    assert bench.max_over_ranks(7.25, 1, "cpu") == 7.25
    assert bench.job_gbs(2.0e9, 10, 1, 1000.0) == pytest.approx(20.0)


def test_reference_arm_rank0_line_shape():
    args = type("A", (), {"reference_rows": 2, "warmup": 3, "steps": 1})()
    line = bench.run_reference(args, 0, 1)
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert torch.__version__  # the arm needs no GPU
