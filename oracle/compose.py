"""Workload-level compositions of the oracle steps (test infrastructure only).

Each function rebuilds, from the seeded generator alone, exactly the inputs
one query of a workload sees, packs them with the oracle's own packers and runs
the oracle steps in the pages' order:

* Full layer [study, lightning-indexer note]: score every visible entry,
  take the top-512, attend over those entries plus the SWA window.
* Reindex layer [study, lightning-indexer note: decoder Reindex layers score
  only a 16,384-position pool picked earlier as blocks of 8]: the Full layer's scores
  pick 2,048 blocks of 8; the Reindex layer's own indexer query scores only
  those positions and takes the top-512 among them.

Nothing here reads a GPU result.
"""
from __future__ import annotations

import functools

import numpy as np

from gen.workloads import Workload, TOPK, SWA, BLOCK, POOL_BLOCKS

__all__ = ["packed_keys", "kv_records", "swa_records", "query_inputs", "decode_query",
           "full_scores", "reindex_query", "reindex_on_pool"]


def _o():
    import oracle
    return oracle


@functools.lru_cache(maxsize=4)
def _packed_keys_cached(wl_key, seq: int, n: int):
    wl = _WL[wl_key]
    o = _o()
    out = np.zeros((n, o.IDX_BYTES), np.uint8)
    step = 1 << 16
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        out[r0:r1] = o.pack_idx(wl.key_rows(seq, np.arange(r0, r1)))
    return out


_WL = {}


def _wkey(wl: Workload):
    k = (wl.name, wl.seed, wl.n_entries, wl.n_seq, wl.zipf, wl.m)
    _WL[k] = wl
    return k


def packed_keys(wl: Workload, seq: int, n: int) -> np.ndarray:
    """Oracle-packed logical 68-byte indexer keys of entries [0, n) of a sequence."""
    return _packed_keys_cached(_wkey(wl), seq, n)


def kv_records(wl: Workload, seq: int, entries) -> np.ndarray:
    """Oracle-packed 288-byte latent records of the given entries (m=1 or m=2)."""
    o = _o()
    entries = np.asarray(entries, dtype=np.int64)
    if entries.size == 0:
        return np.zeros((0, o.KV_BYTES), np.uint8)
    if wl.m == 1:
        return o.pack_kv(wl.latent_rows(seq, entries))
    tok = np.stack([2 * entries, 2 * entries + 1], axis=1).reshape(-1)
    pooled = o.pool_m2(wl.latent_rows(seq, tok), wl.gate_rows(seq, tok))
    return o.pack_kv(pooled)


def swa_records(wl: Workload, seq: int, first: int, cnt: int) -> np.ndarray:
    o = _o()
    slots = (first + np.arange(cnt, dtype=np.int64)) % wl.swa_cap
    if cnt == 0:
        return np.zeros((0, o.SWA_BYTES), np.uint8)
    return o.pack_swa(wl.swa_rows(seq, slots))


def query_inputs(wl: Workload, qi: int, reindex: bool = False):
    o = _o()
    return o.pack_idx(wl.qidx(qi, reindex)), wl.w(qi, reindex)


def full_scores(wl: Workload, qi: int, reindex: bool = False) -> np.ndarray:
    """fp64 indexer scores of every visible entry of query qi's sequence."""
    o = _o()
    seq, n = int(wl.q_seq()[qi]), int(wl.n_vis()[qi])
    qidx, w = query_inputs(wl, qi, reindex)
    return o.index_score(packed_keys(wl, seq, n), qidx, w)


def _attend(wl: Workload, qi: int, sel: np.ndarray, out_fp64=True):
    o = _o()
    seq = int(wl.q_seq()[qi])
    valid = sel[sel >= 0]
    kv = kv_records(wl, seq, valid)
    sw = swa_records(wl, seq, int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi]))
    return o.sparse_attn(wl.q(qi), kv, sw, int(wl.pos()[qi]))


def decode_query(wl: Workload, qi: int, k: int = TOPK) -> dict:
    """Full-layer decode of query qi: scores, top-k selection, attention output."""
    o = _o()
    s = full_scores(wl, qi)
    sel = o.topk(s, k)
    return {"scores": s, "sel": sel, "out": _attend(wl, qi, sel)}


def reindex_on_pool(wl: Workload, qi: int, blocks, k: int = TOPK) -> dict:
    """The Reindex layer's own step for query qi over a given pool of 8-entry
    blocks (block ids, -1 = none): its indexer query scores the pool's visible
    positions, and the top-k of those scores (lower position first on ties,
    positions ascending) is the selection."""
    o = _o()
    seq, n = int(wl.q_seq()[qi]), int(wl.n_vis()[qi])
    blocks = np.asarray(blocks)
    vb = np.sort(blocks[blocks >= 0].astype(np.int64))
    pos = (vb[:, None] * BLOCK + np.arange(BLOCK)[None, :]).reshape(-1)
    pos = pos[pos < n]
    qidx, w = query_inputs(wl, qi, reindex=True)
    s_pool = o.index_score(packed_keys(wl, seq, n)[pos], qidx, w)
    loc = o.topk(s_pool, k)
    sel = np.where(loc >= 0, pos[np.maximum(loc, 0)], -1).astype(np.int32)
    return {"pool_pos": pos, "scores_pool": s_pool, "sel": sel}


def reindex_query(wl: Workload, qi: int, k: int = TOPK) -> dict:
    """Reindex-layer decode of query qi: Full-layer scores -> 2,048-block pool ->
    Reindex scores over the pool's positions -> top-k -> attention."""
    o = _o()
    s_full = full_scores(wl, qi)
    blocks = o.pool_blocks(s_full, BLOCK, POOL_BLOCKS)
    r = reindex_on_pool(wl, qi, blocks, k)
    return {"scores_full": s_full, "blocks": blocks, "pool_pos": r["pool_pos"], "scores_pool": r["scores_pool"],
            "sel": r["sel"], "out": _attend(wl, qi, r["sel"])}
