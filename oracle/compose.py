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
           "full_scores", "reindex_query", "reindex_on_pool", "decoder_step_query", "layer_attention", "build_cache"]


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


def reindex_on_pool(wl: Workload, qi: int, blocks, k: int = TOPK, layer: int = 0) -> dict:
    """The Reindex layer's own step for query qi over a given pool of 8-entry
    blocks (block ids, -1 = none): its indexer query scores the pool's visible
    positions, and the top-k of those scores (lower position first on ties,
    positions ascending) is the selection.  layer: which Reindex layer's query
    and weights (0: the single Reindex layer of the Reindex workload; 1..4:
    the decoder step's Reindex layers)."""
    o = _o()
    seq, n = int(wl.q_seq()[qi]), int(wl.n_vis()[qi])
    blocks = np.asarray(blocks)
    vb = np.sort(blocks[blocks >= 0].astype(np.int64))
    pos = (vb[:, None] * BLOCK + np.arange(BLOCK)[None, :]).reshape(-1)
    pos = pos[pos < n]
    if layer == 0:
        qidx, w = query_inputs(wl, qi, reindex=True)
    else:
        qidx, w = o.pack_idx(wl.qidx_reindex(qi, layer)), wl.w_reindex(qi, layer)
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


def layer_attention(wl: Workload, qi: int, layer: int, sel) -> np.ndarray:
    """Attention of decoder layer `layer` for query qi over the selection
    `sel` (entry indices, -1 padding) and that layer's own window."""
    o = _o()
    seq = int(wl.q_seq()[qi])
    sel = np.asarray(sel)
    kv = kv_records(wl, seq, sel[sel >= 0])
    first, cnt = int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi])
    slots = (first + np.arange(cnt, dtype=np.int64)) % wl.swa_cap
    sw = o.pack_swa(wl.swa_rows_layer(seq, slots, layer)) if cnt else np.zeros((0, o.SWA_BYTES), np.uint8)
    return o.sparse_attn(wl.q_layer(qi, layer), kv, sw, int(wl.pos()[qi]))


def decoder_step_query(wl: Workload, qi: int, layers, pool=None, sels=None) -> dict:
    """The decoder's layers for query qi in the pages' roles [perchy card
    "Full. Reindex. Reuse."; study, reading notes]: the Full layer scores the
    whole cache, keeps the top-512 and picks the pool of 2,048 blocks of 8;
    each Reindex layer scores the pool with its own indexer query and keeps its
    top-512; each Reuse layer attends over the selection of the selecting
    layer it names.  Every layer attends with its own query and window.
    pool / sels (optional): the pool and the selections to attend over (for
    checking a GPU run's attention on its own selections); by default the
    oracle's.  Returns the pool, the oracle's selections {r: sel} with their
    scores, and the layers' outputs."""
    o = _o()
    s_full = full_scores(wl, qi)
    osel = {0: o.topk(s_full, TOPK)}
    opool = o.pool_blocks(s_full, BLOCK, POOL_BLOCKS)
    use_pool = opool if pool is None else np.asarray(pool)
    scores = {0: (np.arange(s_full.size), s_full)}
    for role, r in layers:
        if role == "reindex" and r not in osel:
            rp = reindex_on_pool(wl, qi, use_pool, layer=r)
            osel[r] = rp["sel"]
            scores[r] = (rp["pool_pos"], rp["scores_pool"])
    att = sels if sels is not None else osel
    outs = [layer_attention(wl, qi, l, att[r]) for l, (role, r) in enumerate(layers)]
    return {"pool": opool, "sel": osel, "scores": scores, "out": outs}


def build_cache(tokens_bf16: np.ndarray, gate_logits, w_idx_bf16: np.ndarray, m: int) -> dict:
    """The cache a prompt's tokens leave (encoder entries: m = 2, two tokens
    pooled into one entry by the learned softmax gate; decoder: m = 1), in the
    pages' order ("An infra-oriented diagram of the DeepSeek-V4.1-Flash
    architecture", reading notes on the Full layer's global KV and section "The
    KV cache"): the entry's latent, its 288-B main-cache record, its indexer key
    (the 512 -> 128 projection of the same latent) and that key's 68-B record."""
    o = _o()
    lat = np.asarray(tokens_bf16, np.uint16).reshape(-1, 512)
    if m == 2:
        lat = o.pool_m2(lat, gate_logits)
    keys = o.project_keys(lat, w_idx_bf16)
    return {"latent": lat, "kv": o.pack_kv(lat), "keys": keys, "idx": o.pack_idx(keys)}
