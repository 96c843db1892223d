"""Multi-rank path of the benchmark on CPU (gloo, world size 2): each rank plans
its own replica batch through the C ABI and the job figure uses the slowest
rank's time.  The decode step itself has no exchange between ranks."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import paged_shared_prefix_gb300 as psp
    import workloads
    case = workloads.make_case("agent", rank, batch=20, tables_only=True)
    step = psp.DecodeStep.for_case(case, num_sms=152)
    step.plan_case(case)
    info = step.plan_info()
    ms_local = 1.0 + rank          # rank 1 is the slower replica
    ms, value = bench.aggregate_replicas(ms_local, 1000, world)
    out[rank] = (ms, value, info["num_splits"])
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 2.0            # slowest rank's time
    assert out[0][1] == pytest.approx(2 * 1000 / 2e-3 / 1e9)
    assert out[0][2] > 0 and out[1][2] > 0
