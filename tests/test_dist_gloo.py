"""The N>1 bookkeeping of the benchmark on CPU: two and four gloo ranks, each
with its own seeded batch, run the oracle's path independently (no data crosses ranks)
and agree on the max step time and the summed token count."""
import os
import socket

import numpy as np
import pytest
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
    import oracle
    from combine_get_dispatch_histograms_gb300 import dist as epdist, inputs
    info = epdist.init_from_env("gloo")
    w = inputs.WORKLOADS["tiny"]
    seed = epdist.rank_seed(0, info.rank)
    x, idx, wts = inputs.make_inputs(w, seed)
    res = oracle.run_normal(x, idx, wts, w.R, w.E, w.num_channels)
    step_time = 1.0 + info.rank  # stand-in per-rank times
    mx = epdist.max_over_ranks(step_time)
    tok = epdist.sum_over_ranks(w.R * w.T)
    epdist.barrier()
    q.put((info.rank, info.world, seed, mx, tok, int(res["notify"]["rank_base"][w.R]),
           res["out"].tobytes()))
    epdist.shutdown()


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks_weak_scaling(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    assert [g[0] for g in got] == list(range(world)) and all(g[1] == world for g in got)
    assert len({g[2] for g in got}) == world            # independent batches
    assert all(g[3] == float(world) for g in got)       # max over ranks of the stand-in times 1..world
    assert all(g[4] == world * 4 * 16 for g in got)     # whole-job tokens
    assert len({g[6] for g in got}) == world            # each rank combined its own tokens


def test_single_process_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    from combine_get_dispatch_histograms_gb300 import dist as epdist
    info = epdist.init_from_env("gloo")
    assert (info.rank, info.world) == (0, 1)
    assert epdist.max_over_ranks(3.5) == 3.5 and epdist.sum_over_ranks(7) == 7
