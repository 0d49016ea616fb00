"""The multi-rank host logic of bench.py on two gloo ranks (CPU): each rank
verifies an independent batch, the reported time is the slowest rank's, and
the value counts the work of every rank.  The verification itself runs on the
oracle here, so the test needs no GPU."""
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    import oracle
    import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = synth.chain_tiny(seed=bench.rank_seed(rank), R=3, gamma=4, V=64)
    res = oracle.verify_chain(case.target.f64, case.draft.f64, case.tokens, case.uniforms, 1.0)
    ms_local = 1.0 + rank                       # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms_local, dist, torch.device("cpu"))
    rate = bench.whole_job_rate(3 * 4, world, ms_max)
    # every rank sees the same aggregate and each rank's batch is its own
    toks = torch.tensor(case.tokens.astype(np.int64).ravel())
    gathered = [torch.zeros_like(toks) for _ in range(world)]
    dist.all_gather(gathered, toks)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, ms_max, rate, int(res.accepted.sum()), [g.tolist() for g in gathered]))


def test_two_gloo_ranks_weak_scaling():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    for rank, ms_max, rate, _, _ in results:
        assert ms_max == 2.0                    # the slowest rank's time everywhere
        assert rate == pytest.approx(2 * 12 / 2e-3)
    gathered = results[0][4]
    assert gathered[0] != gathered[1]           # independent batches per rank
