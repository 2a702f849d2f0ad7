"""The benchmark's multi-process path on CPU: two ranks over gloo, as torchrun
launches them (one process per GPU, no data-path collective).  Checks the
rendezvous, the barrier, the max-over-ranks timing and that the reference arm
does its work on rank 0 only."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    bench = _load_bench()
    r, w, local = bench.dist_init()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + rank, w, "cpu")

    class Args:
        steps, warmup = 1, 0

    called = []
    bench.oracle_sample = lambda *a, **k: called.append(1) or {"mla_tflops": 1.0, "idx_tokens_per_s": 1.0,
                                                                 "mla_s": 1.0, "idx_s": 1.0}
    bench.run_reference(Args, r, w)
    import torch.distributed as dist

    dist.destroy_process_group()
    out.put((rank, m, len(called)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_replica_helpers_over_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    assert res[0][1] == res[1][1] == 11.0          # max over ranks
    assert res[0][2] == 1 and res[1][2] == 0       # reference arm: rank 0 does its one step, rank 1 exits
