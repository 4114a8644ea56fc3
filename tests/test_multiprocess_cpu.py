"""The N > 1 path of bench.py, on CPU: two gloo ranks.

The compressor shards by sequence with no exchange on the data path, so under torchrun each
rank runs its own sequences (weak scaling); the only communication is the barrier around the
timed region and the max over ranks of its duration.  This checks that host logic with a
world of two processes on 127.0.0.1, and that each rank draws different sequences.
"""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import synthetic
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each rank reports its own time; every rank must see the maximum
        t = bench.max_over_ranks(1.5 + rank, world, "cpu")
        # the sequences a rank draws (bench.make_inputs uses sequence index rank * B + b)
        x = synthetic.tokens(1, rank * 1 + 0, 0, 2, 64)
        q.put((rank, t, float(x.sum())))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]
    assert res[0][2] != res[1][2]  # different sequences per rank


def test_reference_arm_runs_on_rank_zero_only():
    import bench
    assert bench.run_reference(type("A", (), {"warmup": 0, "steps": 1})(), rank=1, world=2) is None


def test_clock_record_rejection_rules():
    """A throttled or clock-locked timed region is re-measured; a power cap alone is kept."""
    import bench
    ok = {"sm_mhz": 2050.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.clock_rejection(ok) is None
    assert bench.clock_rejection(None) is None
    assert bench.clock_rejection({**ok, "reasons": ["hw_slowdown", "sw_power_cap"]}) == ["hw_slowdown"]
    assert bench.clock_rejection({**ok, "reasons": ["sw_thermal_slowdown"]}) == ["sw_thermal_slowdown"]
    assert bench.clock_rejection({"sm_mhz": 1100.0, "sm_max_mhz": 2070.0, "reasons": []}) == \
        ["sm_clock_below_max_without_reason"]
    assert bench.clock_rejection({"sm_mhz": 1100.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}) is None
