"""Multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    ms = bench.max_over_ranks(1.0 + rank, w, torch.device("cpu"))
    total = bench.tokens_all_ranks(1000, w)
    q.put((r, w, lr, ms, total))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_timing_and_token_total():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for r, w, lr, ms, total in out:
        assert w == 2 and lr == r
        assert ms == 2.0            # the slowest rank's time
        assert total == 2000        # weak scaling: every rank runs a full replica


def test_traffic_record_is_tied_to_the_kernel_sources(monkeypatch):
    import bench
    import synthetic as syn
    w = syn.WORKLOADS[bench.DEFAULT_WORKLOAD]   # the headline workload is always recorded
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as fh:
        rec = __import__("json").load(fh)
    if rec.get("_kernel_sources_sha256") == bench.kernel_sources_digest():
        assert bench.load_traffic(w, "fused") == rec[f"{w.name}|fused"]
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "changed")
    assert bench.load_traffic(w, "fused") is None
