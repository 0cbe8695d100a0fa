"""The N > 1 launch path of bench.py on CPU (gloo, world size 2, no GPU): ranks join through the
environment torch.distributed.run sets, agree on the slowest rank's step time, and report the
whole-job value of weak scaling (each rank runs its own copy of the workload; the linear layer
needs no data-path collective).  The reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    ms = bench.max_over_ranks(w, 10.0 + 5.0 * r)        # rank 1 is the slow one
    value = bench.whole_job_tflops(1e12, w, ms)
    out.put((r, local, ms, value))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_ranks_agree_on_slowest_time_and_whole_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    assert all(local == r for r, local, _, _ in res)
    assert all(ms == 15.0 for _, _, ms, _ in res)          # max over ranks
    # 2 ranks x 1 TFLOP per step in 15 ms
    assert all(v == pytest.approx(2 * 1e12 / 15e-3 / 1e12) for *_, v in res)


def _leaving_rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import time
    import bench
    w, r, _ = bench.dist_setup(timeout_s=10.0)
    if r == 1:
        os._exit(3)                                     # leaves between steps, no collective in flight
    t0 = time.monotonic()
    try:
        bench.barrier(w)
        out.put((r, "no error", time.monotonic() - t0))
    except Exception as e:                              # the surviving rank learns of it on the host
        out.put((r, type(e).__name__, time.monotonic() - t0))


def test_a_rank_that_leaves_ends_the_others_barrier_with_an_error():
    """Failure detection on the host: rank 1 exits after joining; rank 0's next barrier raises
    within the process-group timeout instead of waiting forever."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_leaving_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    r, outcome, waited = out.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
    assert r == 0 and outcome != "no error"
    assert waited < 60.0
    assert procs[1].exitcode == 3 and procs[0].exitcode == 0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench
    # a non-zero rank returns at once, prints nothing and needs no oracle work
    assert bench.run_reference(None, 2, 1) is None
    assert capsys.readouterr().out == ""
