"""bench.py's job accounting on CPU.

Under torchrun every rank decodes its own replica of the workload (requests are
independent; no data-path collective): the job time is the slowest rank's time
and the job throughput counts all ranks' bytes.  Checked here with the gloo
backend at world size 2, plus the gate that keeps a recorded ncu traffic figure
only while the kernel sources it was taken on are unchanged.
"""
import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max_time(times[rank], dist, "cpu")
        v = bench.job_throughput(250e6, 100, world, t)
        dist.barrier()
        out_q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_bytes_add_up():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect_v = 250e6 * 100 * 2 / 0.020 / 1e9
    for rank, t, v in res:
        assert t == 20.0
        assert v == pytest.approx(expect_v)


def test_single_rank_accounting():
    import bench
    assert bench.reduce_max_time(7.0) == 7.0
    assert bench.job_throughput(1e9, 10, 1, 1000.0) == pytest.approx(10.0)


def test_recorded_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    import bench
    with open(bench.TRAFFIC_RECORD) as f:
        rec = json.load(f)
    assert rec["records"]
    for r in rec["records"]:
        step = 2 * r["algorithmic_bytes"]
        t = bench.recorded_traffic(step, r["applies_to"], "auto")
        if t is not None:   # sources unchanged since the capture
            assert t == pytest.approx(2 * (r["dram_bytes_read"] + r["dram_bytes_write"]))
        assert bench.recorded_traffic(step, r["applies_to"], "simt") is None
    assert bench.recorded_traffic(1e9, "some-other-workload", "auto") is None
    stale = dict(rec, sources_sha256="0" * 64)
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(stale))
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(p))
    r = rec["records"][0]
    assert bench.recorded_traffic(2 * r["algorithmic_bytes"], r["applies_to"], "auto") is None
