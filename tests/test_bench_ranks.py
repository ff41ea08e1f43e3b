"""Host logic of bench.py's multi-rank mode, on CPU with the gloo backend (world size 2).

Ranks are replicas (each holds the full per-GPU workload: weak scaling); the
job's time is the slowest rank's and the job's rate counts every rank's units.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0])
    # the re-measure decision is rank 0's, whatever the other ranks would have said
    agreed = (bench.agree_over_ranks(rank == 0), bench.agree_over_ranks(rank == 1))
    out.put((rank, (got, agreed)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == [2.0, 10.0, 5.0]
    assert res[0][1] == res[1][1] == (True, False)


def test_single_process_passthrough_and_rate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]
    # 2 ranks x 10 steps x 5 units in 2 s (slowest rank) = 50 units/s
    assert bench.job_rate(5, 2, 10, 2.0) == 50.0


def test_clock_record_rejection_rule():
    """A slowdown reason, or an SM clock well below its maximum with no reason, disqualifies a timed
    region; a power cap alone does not."""
    sys.path.insert(0, ROOT)
    import bench
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1700.0, reasons=["sw_power_cap"]))
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[r]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1500.0))
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1990.0))
    assert not bench.clocks_rejected(None)
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]})
    assert bench.agree_over_ranks(True) and not bench.agree_over_ranks(False)
