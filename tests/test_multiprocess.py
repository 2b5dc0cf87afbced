"""The bench's multi-replica host logic on CPU, world size 2 over gloo (no GPU).

SageBwd attention shards over (batch, kv head) with no exchange, so several
GPUs run independent replicas: the only cross-rank step of the bench is the
maximum of the step times, from which rank 0 reports whole-job throughput.
The reference arm runs on rank 0 only; the other ranks exit without output.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, e2e = bench.max_over_ranks([4.0 + rank, 5.0 - rank], dist, "cpu")
    out[rank] = (ms, e2e, bench.whole_job_tops(2.0e12, ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_step_times_take_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, e2e, tops = out[rank]
        assert (ms, e2e) == (5.0, 5.0)  # [4, 5] and [5, 4]: the maximum of each
        assert abs(tops - 2 * 2.0e12 / 5e-3 / 1e12) < 1e-9  # both replicas' work in the slowest time


def test_reference_arm_prints_only_on_rank_0(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from bit_trainable_attention_gb300 import workloads as W
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(None, W.WORKLOADS["tiny"]) is None
    assert buf.getvalue() == ""
