"""World-size-2 gloo check of the replica timing logic on CPU: each rank runs
its own independent problem (here: the oracle on its own seed), the elapsed
time is max-reduced, and the whole-job rate counts every rank's units."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import oracle
    from frame_wise_gated_forward_b300 import inputs, replicas
    r, lr, w = replicas.init("gloo")
    x = inputs.draw(1, 2, 3, 16, 32, 32, seed=100 + r)
    res = oracle.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], None,
                               B=1, H=2, F=3, N=16, dk=32, dv=32, n_threads=1)
    replicas.barrier()
    t_local = 1.0 + r            # pretend rank r took 1 + r seconds
    t_max = replicas.max_over_ranks(t_local)
    units = replicas.sum_over_ranks(48)
    rate = replicas.throughput(48, 10, t_max, w)
    q.put((r, w, t_max, units, rate, float(np.abs(res["state"]).sum())))
    replicas.shutdown()


def test_two_rank_gloo_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    outs = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in outs] == [2, 2]
    assert all(o[2] == 2.0 for o in outs)          # max over ranks
    assert all(o[3] == 96.0 for o in outs)         # units summed over ranks
    assert all(abs(o[4] - 48 * 10 * 2 / 2.0) < 1e-9 for o in outs)
    assert outs[0][5] != outs[1][5]                # independent problems per rank


def test_single_process_defaults():
    from frame_wise_gated_forward_b300 import replicas
    assert replicas.max_over_ranks(3.5) == 3.5
    assert replicas.throughput(100, 4, 2.0, 1) == 200.0
