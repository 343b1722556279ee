"""The N > 1 logic of bench.py on CPU: two gloo ranks (spawned processes).

Requests are independent, so ranks never exchange data on the path; the only
cross-rank steps are the barriers around the timed region and the max of the
per-rank step times.  Each rank draws its own seeded batch.
"""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    from tree_speculative_decoding_tsd_gb300 import workloads as W
    d = bench.Dist()
    try:
        d.barrier()
        mx = d.max(float(10 + rank))
        w0 = W.WORKLOADS["toy"]
        w = w0.scaled(index=w0.index + 1000 * rank) if rank else w0
        probs = W.draft_probs(w)
        q.put((rank, mx, float(probs.sum()), int(W.root_tokens(w)[0])))
    finally:
        d.close()


def test_two_rank_barrier_max_and_independent_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res[0][1] == res[1][1] == 11.0          # max over ranks seen by both
    # each rank's draft marginals are distributions; the batches differ by rank
    assert abs(res[0][2] - 3.0) < 1e-4 and abs(res[1][2] - 3.0) < 1e-4
    assert res[0][3] != res[1][3] or res[0][2] != res[1][2]


def test_single_process_dist_is_a_no_op():
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    d = bench.Dist()
    assert d.world == 1 and d.max(3.5) == 3.5
    d.barrier()
    d.close()
