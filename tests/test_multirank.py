"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own replica (independent sequences, no data-path
collective); the only cross-rank steps are the barrier and the max over the
ranks' times, which these tests exercise with the same functions bench.py
uses."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import ssd_inputs as si
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench._dist()
        assert (r, w) == (rank, world)
        bench._barrier(world)
        ms = 1.0 + rank  # rank 1 is the slower one
        ms_max = bench._max_over_ranks(ms, world, device="cpu")
        value = bench.whole_job_tokens_per_s(world, si.PREFILL, ms_max)
        # every rank draws different sequences
        a = si.prefill_inputs(si.TINY, seed=bench.rank_seed(rank), act_dtype=torch.float32)
        gathered = [torch.zeros_like(a["xbc"]) for _ in range(world)]
        dist.all_gather(gathered, a["xbc"])
        out[rank] = (ms_max, value, bool(torch.equal(gathered[0], gathered[1])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_value():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    import ssd_inputs as si
    for r in range(world):
        ms_max, value, same = out[r]
        assert ms_max == pytest.approx(2.0)
        assert value == pytest.approx(2 * si.PREFILL.seqlen / 2e-3)
        assert not same
