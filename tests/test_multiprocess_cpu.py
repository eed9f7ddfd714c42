"""The replicas-only multi-GPU path of bench.py, exercised with two gloo ranks on
the CPU: rendezvous on 127.0.0.1, barrier, max-over-ranks timing, the
whole-job throughput of N independent replicas, and the reference arm running
on rank 0 only (the other ranks exit without work or output)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import argparse

    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + rank, w)  # rank r "took" 10 + r ms
    value = bench.replica_throughput(w, 8192, 5, slowest)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.run_reference(argparse.Namespace(ref_tokens=4, warmup=3, steps=1, gpus=w), w, r) if r else 0
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((rank, slowest, value, rc, buf.getvalue()))


def test_two_gloo_ranks_replicas_timing_and_reference_arm_rank0_only():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, rc, printed in res:
        assert slowest == 11.0                       # the slowest rank sets the time
        assert value == pytest.approx(2 * 8192 * 5 / 0.011)  # whole-job tokens/s over both replicas
        assert rc == 0
    assert res[1][4] == ""                           # rank 1: no work, no output
