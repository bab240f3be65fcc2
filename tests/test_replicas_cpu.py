"""The benchmark's multi-process path on CPU: two gloo ranks.

Multi-GPU runs are independent replicas (the hot path has no exchange step);
what the ranks share is the rendezvous, a barrier around the timed region, the
max-over-ranks time and rank 0 alone reporting. These run here as two spawned
gloo processes on 127.0.0.1.
"""

import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    try:
        w, r, _ = bench.dist_setup(world)
        bench.barrier(w)
        slowest = bench.max_over_ranks(10.0 + 5.0 * r, w, torch.device("cpu"))
        # the reference arm: ranks other than 0 leave without work
        ref_rc = bench.run_reference(None, None, None, w, r) if r != 0 else None
        bench.barrier(w)
        q.put((r, w, slowest, ref_rc))
    finally:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in procs:
            r, w, slowest, ref_rc = q.get(timeout=120)
            results[r] = (w, slowest, ref_rc)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert sorted(results) == [0, 1]
    assert all(w == 2 and slowest == 15.0 for w, slowest, _ in results.values())
    assert results[1][2] == 0
    assert all(p.exitcode == 0 for p in procs)


def test_single_process_needs_no_rendezvous():
    import bench
    old = {k: os.environ.pop(k, None) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    try:
        assert bench.dist_setup(1) == (1, 0, 0)
        assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    finally:
        for k, v in old.items():
            if v is not None:
                os.environ[k] = v
