"""Multi-rank aggregation of bench.py on CPU with gloo (world size 2).

Every rank runs an independent replica of the decode workload; the job's throughput is
all ranks' units over the slowest rank's time.  Each rank's kernels never wait on
another rank, so the N>1 path is exercised here without a GPU.
"""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.aggregate_ranks(10.0 + 5.0 * rank, 100 * (rank + 1), device="cpu")
    # a clock rejection on one rank makes every rank measure again
    again = bench.any_rank(rank == 1, device="cpu")
    q.put((rank, ms, units, again))
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, units, again in res:
        assert ms == 15.0 and units == 300
        assert again is True


def test_aggregate_single_process_passthrough():
    import bench
    assert bench.aggregate_ranks(3.5, 7) == (3.5, 7)


def test_clock_rejection_rule():
    import bench
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, reasons=["sw_power_cap"]))          # kept, noted
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1500.0, reasons=["sw_power_cap"]))
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[r]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1200.0))                         # a leftover lock
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]})
    assert bench.any_rank(True) and not bench.any_rank(False)                    # single process
