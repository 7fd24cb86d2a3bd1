"""The host logic of a multi-GPU run (bench.py under torchrun), on two gloo
ranks on the CPU: each rank decodes a batch of its own, the barrier holds every
rank, the job's time is its slowest rank's, and its rate counts every rank's
units.  (Decode batches are independent: the ranks are replicas, with no
collective on the data path.)"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import time
    import numpy as np
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from compressed_sparse_attention_index_gb300 import ranks
        from gen.workloads import CONFIGS
        r, w, lr = ranks.rank_env()
        wl = ranks.rank_workload(CONFIGS[4], r)
        q_sig = int(np.asarray(wl.q(0)).view(np.uint16)[:4096].astype(np.int64).sum())
        # rank 1 arrives late: the barrier must hold rank 0 until it does
        if r == 1:
            time.sleep(0.5)
        t0 = time.time()
        ranks.barrier()
        waited = time.time() - t0
        ms = ranks.max_over_ranks(10.0 + 5.0 * r)             # rank r's timed region took 10 + 5 r ms
        rate = ranks.whole_job_rate(8 * 3, w, ms)             # 8 queries x 3 steps per rank
        rows = [None] * w
        dist.all_gather_object(rows, (r, w, lr, wl.name, wl.seed, wl.n_entries, q_sig, waited, ms, rate))
        if r == 0:
            out.put(rows)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        rows = q.get(timeout=120)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    (r0, w0, lr0, name0, seed0, n0, sig0, wait0, ms0, rate0), (r1, w1, lr1, name1, seed1, n1, sig1, wait1, ms1, rate1) = rows
    assert (r0, r1, w0, w1, lr0, lr1) == (0, 1, 2, 2, 0, 1)
    assert name0 == "long_full_decode_N1M_B8_zipf" and name1 != name0      # rank 0 keeps the configuration
    assert seed0 != seed1 and n0 == n1 and sig0 != sig1                    # same shapes, its own batch
    assert wait0 >= 0.3 > wait1                                            # the barrier held rank 0
    assert ms0 == ms1 == 15.0                                              # the slowest rank's time, on every rank
    assert rate0 == rate1 == pytest.approx(2 * 8 * 3 / 15e-3)              # every rank's units


def test_one_rank_is_unchanged():
    from compressed_sparse_attention_index_gb300 import ranks
    from gen.workloads import CONFIGS
    assert ranks.rank_workload(CONFIGS[4], 0) is CONFIGS[4]
    assert ranks.max_over_ranks(12.5) == 12.5                               # no process group: local value
    assert ranks.whole_job_rate(24, 1, 12.0) == pytest.approx(2000.0)
