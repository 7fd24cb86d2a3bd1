"""Sequence sharding (entries of one cache split over ranks), checked on CPU
ranks against the unsharded oracle: the top-k of the union of the ranks' local
top-k lists is the global top-k, and the log-sum-exp merge of the ranks'
attention outputs is the attention over all the selected entries."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("ranks", [2, 3, 7])
def test_merge_topk_equals_global_topk(oracle_lib, ranks):
    rng = np.random.default_rng(40 + ranks)
    n, k = 5000, 512
    s = rng.standard_normal(n)
    s[rng.choice(n, 400, replace=False)] = 0.75    # ties, many of them across shard boundaries
    s[:50] = -0.0
    from compressed_sparse_attention_index_gb300 import shard
    lists_s, lists_i = [], []
    for lo, hi in shard.shard_ranges(n, ranks):
        loc = oracle_lib.topk(s[lo:hi], k)
        loc = loc[loc >= 0].astype(np.int64)
        lists_s.append(s[lo:hi][loc])
        lists_i.append(loc + lo)
    assert np.array_equal(shard.merge_topk(lists_s, lists_i, k), oracle_lib.topk(s, k))


def test_merge_topk_short_union_pads():
    from compressed_sparse_attention_index_gb300 import shard
    got = shard.merge_topk([[1.0, 2.0], [2.0]], [[7, 3], [1]], 5)
    assert got.tolist() == [1, 3, 7, -1, -1]       # equal scores: the lower index first; all kept


def test_lse_merge_of_a_split_softmax(oracle_lib):
    """Splitting a softmax's entries into parts and merging their outputs by
    log-sum-exp gives the softmax over all of them (oracle attention)."""
    from gen.workloads import small
    from oracle.compose import kv_records, swa_records
    from compressed_sparse_attention_index_gb300 import shard
    wl = small(n_seq=1, n_entries=2000, seed=310)
    sel = oracle_lib.decode_query(wl, 0)["sel"]
    sel = sel[sel >= 0]
    swa = swa_records(wl, 0, int(wl.swa_first()[0]), int(wl.swa_cnt()[0]))
    ref = oracle_lib.sparse_attn(wl.q(0), kv_records(wl, 0, sel), swa, int(wl.pos()[0]))
    parts = [sel[:100], sel[100:101], sel[101:], sel[:0]]        # one part empty
    outs, lses = [], []
    for j, p in enumerate(parts):
        o, l = oracle_lib.sparse_attn_lse(wl.q(0), kv_records(wl, 0, p), swa if j == 0 else swa[:0],
                                          int(wl.pos()[0]))
        outs.append(o)
        lses.append(l)
    assert np.isneginf(lses[3]).all() and not np.any(outs[3])
    got = shard.lse_merge(outs, lses)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import oracle as oracle_lib
    from gen.workloads import small
    from oracle.compose import kv_records, swa_records
    from compressed_sparse_attention_index_gb300 import shard
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = small(n_seq=1, n_entries=6000, seed=320)
        n = int(wl.n_vis()[0])
        lo, hi = shard.shard_ranges(n, world)[rank]
        scores = oracle_lib.full_scores(wl, 0)[:n]        # this rank's range is all it uses
        loc = oracle_lib.topk(scores[lo:hi], 512)
        loc = loc[loc >= 0].astype(np.int64)
        lists = [None] * world
        dist.all_gather_object(lists, (scores[lo:hi][loc], loc + lo))          # the one all-gather
        sel = shard.merge_topk([x[0] for x in lists], [x[1] for x in lists], 512)
        mine = sel[(sel >= lo) & (sel < hi)]
        swa = swa_records(wl, 0, int(wl.swa_first()[0]), int(wl.swa_cnt()[0]))
        o, lse = oracle_lib.sparse_attn_lse(wl.q(0), kv_records(wl, 0, mine), swa if rank == 0 else swa[:0],
                                            int(wl.pos()[0]))
        parts = [None] * world
        dist.all_gather_object(parts, (o, lse))                                 # the LSE-merge exchange
        if rank == 0:
            out.put((sel, shard.lse_merge([p[0] for p in parts], [p[1] for p in parts])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_one_cache(oracle_lib):
    import torch.multiprocessing as mp
    from gen.workloads import small
    from oracle.compose import kv_records, swa_records
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        sel, out = q.get(timeout=180)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    wl = small(n_seq=1, n_entries=6000, seed=320)
    ref = oracle_lib.decode_query(wl, 0)
    assert np.array_equal(sel, ref["sel"])                     # the exact global top-512
    assert np.max(np.abs(out - ref["out"])) <= 1e-12 * np.max(np.abs(ref["out"]))
