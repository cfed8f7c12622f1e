"""The N > 1 bench path on CPU: two gloo ranks agree on the slowest rank's
time (max over ranks) and on the whole-job value (all ranks' work over that
time).  No GPU; rendezvous on 127.0.0.1."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r measured (r + 1) ms for the step and (3 - r) ms for attention
    step, attn = bench.max_over_ranks([rank + 1.0, 3.0 - rank], "cpu")
    value = bench.whole_job_tflops(2e12, world, attn)
    dist.barrier()
    out[rank] = (step, attn, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        step, attn, value = out[r]
        assert step == 2.0
        assert attn == 3.0
        assert value == pytest.approx(2e12 * 2 / 3e-3 / 1e12)


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]
    assert bench.whole_job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)
