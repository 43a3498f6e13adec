"""Host-side logic of bench.py's multi-process path on CPU: two gloo ranks,
as torchrun would start them (127.0.0.1 rendezvous). Every rank decodes its
own disjoint token stream (weak scaling, no data-path collective); the job's
time is the maximum over ranks and its throughput all ranks' tokens over that
time."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from bit_codebook_quantized_dequant_gb300 import synth as S


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench._dist()
    times = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]  # this rank's timed regions (ms)
    ms, ms_e2e = bench.max_over_ranks(times, dist)
    start = bench.rank_token_start(r, 8)
    x = S.tokens(S.workload_seed("tiny-decode"), S.WORKLOADS["tiny-decode"], 8, start=start)
    out[rank] = (ws, r, local, ms, ms_e2e, start, x.tobytes())
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ws, r, local, ms, ms_e2e, start, _ = res[rank]
        assert (ws, r, local) == (world, rank, rank)
        assert ms == 15.0 and ms_e2e == 20.0  # max over ranks, on every rank
        assert start == 8 * rank
    # disjoint token streams: rank 1's tokens are the continuation of rank 0's
    x0 = np.frombuffer(res[0][6], dtype=np.uint16)
    x1 = np.frombuffer(res[1][6], dtype=np.uint16)
    both = S.tokens(S.workload_seed("tiny-decode"), S.WORKLOADS["tiny-decode"], 16).ravel()
    np.testing.assert_array_equal(np.concatenate([x0, x1]), both)
    # whole-job throughput: all ranks' units over the slowest rank's time
    assert bench.job_throughput(world, 1000, 15.0) == pytest.approx(2 * 1000 / 0.015)


def test_single_process_defaults():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench._dist() == (1, 0, 0)
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]


def test_prefill_cpu_baseline_on_a_tiny_workload():
    # the oracle's prefill rate reported beside each prefill section
    cb = bench.cpu_baseline_prefill("tiny-decode", tokens=3)
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["unit"] == "tok/s"
    assert cb["value"] > 0 and "first 3 tokens" in cb["sample"]
