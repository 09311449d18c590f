"""The bench's multi-rank host logic on CPU: two gloo ranks (one process per
rank, as the launcher would start them). Replicas only -- no data-path
collective exists -- so what is checked is the timing reduction (max over
ranks) and that only rank 0 does the reference arm's work."""
import os
import socket
import types

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, root, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, root)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got = bench.max_over_ranks({"decode": 1.0 + rank, "prefill": 10.0 - rank}, ws)

        def no_work(*a, **k):
            raise AssertionError("the oracle ran on a rank other than 0")
        if rank != 0:
            bench.cpu_oracle_decode = no_work
            bench.run_reference(types.SimpleNamespace(steps=1, warmup=3, ref_budget=0.1))
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank0_only_reference():
    ws = 2
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, root, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=10) for _ in range(ws))
    for r in range(ws):
        assert results[r] == {"decode": 2.0, "prefill": 10.0}
