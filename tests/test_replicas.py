"""Host-side replica plumbing with two gloo ranks on the CPU: barrier, max of
the elapsed time and whole-job throughput."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from mask_aware_exact_gb300 import replicas as R
    assert R.init("gloo")
    R.barrier()
    # rank r processed (r+1) * 10 units in (r+1) seconds
    agg = R.aggregate_throughput((rank + 1) * 10.0, float(rank + 1))
    q.put((rank, agg))
    R.finalize()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    for r in range(2):
        assert res[r]["total_units"] == 30.0
        assert res[r]["max_elapsed_s"] == 2.0
        assert res[r]["throughput"] == 15.0


def test_single_process_is_identity():
    from mask_aware_exact_gb300 import replicas as R
    os.environ.pop("WORLD_SIZE", None)
    assert not R.init("gloo")
    assert R.aggregate_throughput(5.0, 2.0)["throughput"] == 2.5
