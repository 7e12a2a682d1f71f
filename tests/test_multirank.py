"""The N > 1 path of bench.py on the CPU: two gloo ranks run the benchmark's
distributed plumbing (init, barrier, max over ranks of the timed region, the
whole-job throughput).  The data path has no collective: each rank runs its
own replica of the workload (heads are independent), with its own seed."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import torch.distributed as dist
    r, w = bench._dist_init(world)
    assert (r, w) == (rank, world)
    assert dist.get_backend() == "gloo"
    bench._barrier(w)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    mx = bench._max_over_ranks(ms, w)
    value = bench.job_throughput(1000, w, mx, steps=4)
    # the inputs of the replicas differ (seed + 1000 * rank) but have the same shape
    from fixed_state_recurrent_gb300 import inputs
    q, _, _ = inputs.la_inputs(1, 1, 8, 4, 4, torch.bfloat16, seed=5 + 1000 * rank)
    out[rank] = (mx, value, float(q.float().sum()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_share_the_max_time():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] == out[1][1] == pytest.approx(1000 * 2 * 4 / 15e-3)
    assert out[0][2] != out[1][2]
